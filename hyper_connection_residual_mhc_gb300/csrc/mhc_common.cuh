// mhc_common.cuh -- device helpers and internal launcher declarations shared
// by the libmhc translation units.
#pragma once

#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <stdint.h>

#include <utility>

#include "../../include/mhc.h"

namespace mhc {

constexpr int kHC = MHC_HC;        // residual streams
constexpr int kH = MHC_HIDDEN;     // hidden width
constexpr int kK = MHC_K;          // flattened row width
constexpr int kMix = MHC_MIX;      // mixes per row
constexpr int kChunk = 8;          // bf16 per 16-byte vector
constexpr int kChunksPerStream = kH / kChunk;   // 640

// ---- bf16 <-> fp32 on 16-byte vectors -------------------------------------
// bf16 -> fp32 is exact: the bf16 bits are the top half of the fp32 bits.
__device__ __forceinline__ void unpack8(const uint4 &v, float (&f)[8]) {
  const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    f[2 * q] = __uint_as_float(w[q] << 16);
    f[2 * q + 1] = __uint_as_float(w[q] & 0xFFFF0000u);
  }
}

// fp32 -> bf16, round to nearest even, two at a time (low half = first).
__device__ __forceinline__ uint32_t pack2_rn(float lo, float hi) {
  __nv_bfloat162 b = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t *>(&b);
}

__device__ __forceinline__ uint4 pack8_rn(const float (&f)[8]) {
  uint4 v;
  v.x = pack2_rn(f[0], f[1]);
  v.y = pack2_rn(f[2], f[3]);
  v.z = pack2_rn(f[4], f[5]);
  v.w = pack2_rn(f[6], f[7]);
  return v;
}

// hc_post on one 8-column chunk of a row (deepseek_v4.py, hc_post_torch_impl):
// out_i = bf16( post_i * y + sum_j comb[j][i] * R_j ), fp32 arithmetic in a
// fixed order, one rounding.  cb[j][i] = comb[j][i].
__device__ __forceinline__ void post_chunk(const uint4 (&rv)[kHC], const uint4 &yv,
                                           const float (&pv)[kHC], const float (&cb)[kHC][kHC],
                                           uint4 (&out)[kHC]) {
  float yf[8], rf[kHC][8];
  unpack8(yv, yf);
#pragma unroll
  for (int j = 0; j < kHC; ++j) unpack8(rv[j], rf[j]);
#pragma unroll
  for (int i = 0; i < kHC; ++i) {
    float acc[8];
#pragma unroll
    for (int e = 0; e < 8; ++e) {
      float a = pv[i] * yf[e];
#pragma unroll
      for (int j = 0; j < kHC; ++j) a = fmaf(cb[j][i], rf[j][e], a);
      acc[e] = a;
    }
    out[i] = pack8_rn(acc);
  }
}

// ---- MXFP8: E4M3 codes with a ue8m0 scale per 32 values ---------------------
// (prefill_sp.py, _mxfp8_quantize: per row, per 32 columns.)  The scale rule
// is the OCP Microscaling (MX) v1.0 conversion for E4M3, whose largest
// exponent is 8: e = floor(log2 amax) - 8, clamped below at -127 (a zero or
// tiny block), scale code e + 127; each value becomes E4M3(v / 2^e), rounded
// to nearest-even and saturated to +-448, the sign kept.
constexpr int kMxBlock = 32;
// One block is held by 4 consecutive lanes (lane & ~3 .. | 3), 8 values each
// in column order; v holds the values exactly (bf16 widened).  Every lane of
// the warp must call this together.  Returns the 8 codes (first value in the
// lowest byte) and sets the block's scale code.
__device__ __forceinline__ uint2 mx_block8(const float (&v)[8], uint32_t &scale_code) {
  float amax = 0.f;
#pragma unroll
  for (int e = 0; e < 8; ++e) amax = fmaxf(amax, fabsf(v[e]));
  amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 1));
  amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 2));
  // amax >= 0, so its bits are the biased exponent and the mantissa; a zero
  // or subnormal amax (biased exponent 0) takes the clamp
  const int biased = (int)(__float_as_uint(amax) >> 23);
  const int e = max(biased - 127 - 8, -127);
  scale_code = (uint32_t)(e + 127);
  const float inv = __uint_as_float((uint32_t)(127 - e) << 23);   // 2^-e, exact, normal
  uint32_t w[2];
#pragma unroll
  for (int h = 0; h < 2; ++h) {
    uint16_t p01, p23;
    // cvt ... d, a, b packs a into the high byte and b into the low byte
    asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;"
        : "=h"(p01) : "f"(v[4 * h + 1] * inv), "f"(v[4 * h] * inv));
    asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;"
        : "=h"(p23) : "f"(v[4 * h + 3] * inv), "f"(v[4 * h + 2] * inv));
    w[h] = (uint32_t)p01 | ((uint32_t)p23 << 16);
  }
  return make_uint2(w[0], w[1]);
}

// Streaming (evict-first) 16-byte global accesses for data touched once.
__device__ __forceinline__ uint4 ld_stream(const uint4 *p) { return __ldcs(p); }
// 16 bytes of data that no thread writes during the kernel, without
// allocating an L1 line (a second read of data that L2 still holds)
__device__ __forceinline__ uint4 ld_nc_noalloc(const uint4 *p) {
  uint4 v;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p));
  return v;
}
__device__ __forceinline__ void st_stream(uint4 *p, const uint4 &v) { __stcs(p, v); }

// 1/x for x >= 1e-30 or +inf (the Sinkhorn's sums, each holding eps; 1 +
// exp(-l)): the hardware approximation refined by one Newton step for the
// reciprocal, r + r (1 - x r) with fused multiply-adds, which leaves it
// within about an ulp; 0 where the approximation is 0 (x = inf, or 1/x below
// the normal range), as the IEEE quotient gives.  No branch, so the four
// reciprocals of a Sinkhorn step overlap.
__device__ __forceinline__ float rcp_nr(float x) {
  float r;
  asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(r) : "f"(x));
  return r == 0.f ? 0.f : fmaf(r, fmaf(-x, r, 1.0f), r);
}

// 1/sqrt(x) for x >= 1e-30 or +inf (mean squares plus eps): the hardware
// approximation refined by one Newton step for the reciprocal square root,
// r (3 - x r^2) / 2; 0 for x = inf, as 1/sqrt gives
__device__ __forceinline__ float rsqrt_nr(float x) {
  float r;
  asm("rsqrt.approx.ftz.f32 %0, %1;" : "=f"(r) : "f"(x));
  return r == 0.f ? 0.f : r * fmaf(-0.5f * x * r, r, 1.5f);
}

// ---- programmatic dependent launch -----------------------------------------
// The library's launches carry programmatic stream serialization, so a
// kernel's CTAs may be scheduled while the kernel before it on the stream is
// still running.  Every such kernel calls pdl_wait() before its first global
// memory access: it returns once the grids this one depends on have completed
// and their writes are visible, so stream order holds for any caller.  It then
// calls pdl_trigger(), which lets the next launch schedule its CTAs (they wait
// in turn).  A dependent grid is scheduled only after every CTA of this grid
// has started, so waiting CTAs never hold resources this grid still needs.
// Without the launch attribute both are no-ops.
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_trigger() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// The attribute pays for itself only where a launch carries little work: at
// up to 2048 rows per chunk it takes 2-6 us off a pre + post step (launch
// latency); from 4096 rows on it measured neutral to slightly slower (up to
// +1.5 % replayed from a CUDA graph).  Keyed on the chunk's row count, so all
// shards of a chunk launch alike.
constexpr int64_t kPdlMaxRows = 2048;
inline bool use_pdl(int64_t logical_rows) { return logical_rows <= kPdlMaxRows; }

// host: cudaLaunchKernelEx, with programmatic stream serialization when pdl,
// and a cluster dimension when cluster_x > 1
template <typename... ExpTypes, typename... ActTypes>
inline cudaError_t launch_pdl(void (*kernel)(ExpTypes...), dim3 grid, dim3 block, size_t smem,
                              cudaStream_t s, unsigned cluster_x, bool pdl, ActTypes &&...args) {
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute at[2];
  unsigned n = 0;
  if (pdl) {
    at[n].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    at[n].val.programmaticStreamSerializationAllowed = 1;
    ++n;
  }
  if (cluster_x > 1) {
    at[n].id = cudaLaunchAttributeClusterDimension;
    at[n].val.clusterDim.x = cluster_x;
    at[n].val.clusterDim.y = 1;
    at[n].val.clusterDim.z = 1;
    ++n;
  }
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cfg.attrs = at;
  cfg.numAttrs = n;
  return cudaLaunchKernelEx(&cfg, kernel, std::forward<ActTypes>(args)...);
}

// ---- internal launchers (host side) ----------------------------------------
// Each returns cudaSuccess or the launch error; arguments are validated by the
// C entry points before these are called.
cudaError_t launch_post(const uint16_t *R, const uint16_t *y, const float *post,
                        const float *comb, int64_t rows, int64_t logical_rows, uint16_t *R_out,
                        cudaStream_t s);

cudaError_t launch_combine_norm(const uint16_t *R, const float *pre, const uint16_t *norm_w,
                                float norm_eps, int64_t rows, int64_t logical_rows,
                                uint16_t *x_norm, cudaStream_t s);

// decode-size chunks (logical_rows <= kDecodeMaxRows): all of mhc_pre in one
// launch of 16-CTA clusters, a group of up to 8 rows per cluster, no scratch
// (pre_decode.cu)
constexpr int64_t kDecodeMaxRows = 48;
cudaError_t decode_error_word(unsigned int *out, bool reset);
cudaError_t launch_pre_decode(const uint16_t *R, const float *fn, const float *scale,
                              const float *base, const uint16_t *norm_w, int64_t rows,
                              int64_t logical_rows, const mhc_params &p, uint16_t *x_norm,
                              float *post, float *comb, float *pre_out, float *mix_out,
                              cudaStream_t s, bool fn_stable = false);
// the same launch with hc_post of the previous sublayer first: R_out =
// hc_post(R, y, post_in, comb_in) (mhc_post's bits), then mhc_pre on R_out
cudaError_t launch_post_pre_decode(const uint16_t *R, const uint16_t *y, const float *post_in,
                                   const float *comb_in, const float *fn, const float *scale,
                                   const float *base, const uint16_t *norm_w, int64_t rows,
                                   int64_t logical_rows, const mhc_params &p, uint16_t *R_out,
                                   uint16_t *x_norm, float *post, float *comb, float *pre_out,
                                   float *mix_out, cudaStream_t s, bool fn_stable = false);

// combine + RMSNorm with a fifth warp per row block for the Sinkhorn of the
// comb logits (writes comb [rows, 4, 4])
// mx_q / mx_s non-NULL: the same launch also writes x_norm's MXFP8 codes
// [rows, 5120] and linear ue8m0 scales [rows, 160] (mx_block8 of the bf16
// x_norm values)
cudaError_t launch_combine_norm_sinkhorn(const uint16_t *R, const float *pre,
                                         const uint16_t *norm_w, float norm_eps,
                                         const float *logit, float *comb, float sink_eps,
                                         int iters, int64_t rows, int64_t logical_rows,
                                         uint16_t *x_norm, cudaStream_t s,
                                         uint8_t *mx_q = nullptr, uint8_t *mx_s = nullptr);
// MXFP8 of bf16 rows x [rows, cols] (cols a multiple of 32): codes q [rows,
// cols], linear scales s [rows, cols/32]
cudaError_t launch_mx_quantize(const uint16_t *x, int64_t rows, int64_t cols,
                               int64_t logical_rows, uint8_t *q, uint8_t *s, cudaStream_t st);
// linear scales s [rows, groups] -> the 128x4 tiled layout, ceil(rows/128)*128
// *groups bytes, padding rows zero (groups a multiple of 4)
cudaError_t launch_mx_swizzle(const uint8_t *s, int64_t rows, int64_t groups, uint8_t *out,
                              cudaStream_t st);
// all of hc_head in one pass over R (head_onepass.cu): 4-CTA clusters, fp32
// projections on the CUDA cores, the combine from shared memory.  It is
// latency-bound (a 4-row tile per ~4 us per cluster), so it serves chunks of
// up to 256 rows
constexpr int64_t kHeadOnePassMaxRows = 256;
cudaError_t launch_head_onepass(const uint16_t *R, const float *fn, const float *scale,
                                const float *base, int64_t rows, int64_t logical_rows,
                                float norm_eps, float hc_eps, uint16_t *y, float *pre_out,
                                float *mix_out, cudaStream_t s);
cudaError_t head_error_word(unsigned int *out, bool reset);
// above that: one launch of 16-CTA clusters whose tiles stay in shared
// memory for the combine (head_tile.cu)
cudaError_t launch_head_tile(const uint16_t *R, const float *fn, const float *scale,
                             const float *base, int64_t rows, int64_t logical_rows,
                             float norm_eps, float hc_eps, uint16_t *y, float *pre_out,
                             float *mix_out, cudaStream_t s);
cudaError_t head_tile_error_word(unsigned int *out, bool reset);
// hc_post fused with the next pre's stats (post_pre_fused.cu): writes R_out,
// the next pre's gates to pre_ws [rows, 4], its comb logits to logit_ws
// [rows, 16] and its post gates (+ pre_out, mix_out)
// (fnp: fused_fn_bytes() of scratch for fn in the kernel's B-operand image)
size_t fused_fn_bytes();
// (fn NULL: fnp already holds the image, written by launch_fn_prep_sw64)
cudaError_t launch_post_pre_fused(const uint16_t *R, const uint16_t *y, const float *post,
                                  const float *comb, const float *fn, const float *scale,
                                  const float *base, int64_t rows, int64_t logical_rows,
                                  const mhc_params &p, float *pre_ws, float *logit_ws,
                                  const uint8_t *fnp, uint16_t *R_out, float *post_out,
                                  float *pre_out, float *mix_out, cudaStream_t s);
cudaError_t launch_fn_prep_sw64(const float *fn, uint8_t *fnp, cudaStream_t s, bool pdl);
cudaError_t fused_post_pre_error_word(unsigned int *out, bool reset);

// all of mhc_pre in one launch that reads R from HBM once (pre_onepass.cu):
// 32-row tiles, the four streams of a 64-column block as one MMA operand
// against fn's hi/lo for all four streams, one cluster exchange per tile, the
// combine re-reading its tile from L2.  fn_img NULL: 16-CTA clusters with
// fn's tiles converted into shared memory by the kernel.  fn_img given:
// 16-CTA clusters below kStreamMinRows rows and 8-CTA clusters from there on
// (120 SMs instead of 112), both streaming fn's tile of each block from the
// image beside the block of R.  fn_img: NULL, or fn's
// image of fn_b_img_bytes() (then fn is not read).  mx_q / mx_s non-NULL:
// x_norm's MXFP8 codes [rows, 5120] and linear ue8m0 scales [rows, 160] as
// well.
constexpr int64_t kStreamMinRows = 2048;
cudaError_t launch_pre_onepass(const uint16_t *R, const float *fn, const uint8_t *fn_img,
                               const float *scale, const float *base, const uint16_t *norm_w,
                               int64_t rows, int64_t logical_rows, const mhc_params &p,
                               uint16_t *x_norm, float *post, float *comb, float *pre_out,
                               float *mix_out, cudaStream_t s, uint8_t *mx_q = nullptr,
                               uint8_t *mx_s = nullptr);
// fn [24, 20480] fp32 -> the one-pass kernels' B tiles, laid out for 16 ranks
// of 320 columns (fn_b_img_bytes() bytes); the prepared weights hold one, and
// mhc_pre writes one into its workspace for the streamed build
size_t fn_b_img_bytes();
cudaError_t launch_fn_b_img(const float *fn, uint8_t *img, cudaStream_t s);
cudaError_t onepass_error_word(unsigned int *out, bool reset);
// where the one-pass kernel's expired (0..31) and abandoned (32..63) waits ended
cudaError_t onepass_error_where(unsigned int *out64);

}  // namespace mhc
