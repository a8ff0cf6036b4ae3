// pre_simt.cu -- CUDA-core path of mhc_pre, in three launches:
//   1. stats_partial: partial sums of x.x and x.fn_c over 16 fixed K slices
//   2. finalize     : rsqrt, mix, logits, gates, Sinkhorn (one thread per row)
//   3. combine_norm : y = sum_i pre_i R_i, RMSNorm, bf16 x_norm
// (deepseek_v4.py, DeepseekV4DecoderLayer.hc_pre: hc_pre_torch_impl, then
// hc_split_sinkhorn and the combine; RMSNorm fused as in prefill_sp.py,
// hc_combine_norm_rows).
//
// Every row is reduced in one fixed order that depends on nothing but the
// row's own data: slice boundaries, per-thread strides and the tree of the
// block reductions are compile-time constants.  Row ranges therefore give the
// whole-chunk bits.
#include "mhc_common.cuh"

namespace mhc {
namespace {

constexpr int kSlices = 16;                  // K slices of the stats
constexpr int kSliceK = kK / kSlices;        // 1280
constexpr int kStatsThreads = 256;
constexpr int kStatsRows = 4;                // rows per stats block
constexpr int kPerThreadK = kSliceK / kStatsThreads;   // 5
constexpr int kPartial = kMix + 1;           // 24 dots + sum of squares

static_assert(kSliceK % kStatsThreads == 0, "slice must split evenly");

// partials layout: [slice][row][kPartial] fp32
__global__ void __launch_bounds__(kStatsThreads)
stats_partial_kernel(const uint16_t *__restrict__ R, const float *__restrict__ fn,
                     float *__restrict__ partials, int64_t rows) {
  const int slice = blockIdx.y;
  const int64_t row0 = (int64_t)blockIdx.x * kStatsRows;
  const int tid = threadIdx.x;

  float acc[kStatsRows][kPartial];
#pragma unroll
  for (int r = 0; r < kStatsRows; ++r)
#pragma unroll
    for (int c = 0; c < kPartial; ++c) acc[r][c] = 0.f;

#pragma unroll 1
  for (int s = 0; s < kPerThreadK; ++s) {
    const int k = slice * kSliceK + s * kStatsThreads + tid;
    float x[kStatsRows];
#pragma unroll
    for (int r = 0; r < kStatsRows; ++r) {
      const int64_t m = row0 + r;
      x[r] = m < rows ? __uint_as_float((uint32_t)__ldg(R + m * kK + k) << 16) : 0.f;
      acc[r][kMix] = fmaf(x[r], x[r], acc[r][kMix]);
    }
#pragma unroll
    for (int c = 0; c < kMix; ++c) {
      const float f = __ldg(fn + (int64_t)c * kK + k);
#pragma unroll
      for (int r = 0; r < kStatsRows; ++r) acc[r][c] = fmaf(x[r], f, acc[r][c]);
    }
  }

  // block reduction: warp butterfly, then warps 0..7 in order
  __shared__ float red[kStatsThreads / 32][kStatsRows * kPartial];
  const int lane = tid & 31, warp = tid >> 5;
#pragma unroll
  for (int r = 0; r < kStatsRows; ++r)
#pragma unroll
    for (int c = 0; c < kPartial; ++c) {
      float v = acc[r][c];
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) v += __shfl_xor_sync(0xffffffffu, v, off);
      if (lane == 0) red[warp][r * kPartial + c] = v;
    }
  __syncthreads();
  if (tid < kStatsRows * kPartial) {
    float v = red[0][tid];
#pragma unroll
    for (int w = 1; w < kStatsThreads / 32; ++w) v += red[w][tid];
    const int r = tid / kPartial, c = tid % kPartial;
    const int64_t m = row0 + r;
    if (m < rows) partials[((int64_t)slice * rows + m) * kPartial + c] = v;
  }
}

__device__ __forceinline__ float sigmoidf_(float z) { return 1.0f / (1.0f + expf(-z)); }

__global__ void __launch_bounds__(128)
finalize_kernel(const float *__restrict__ partials, const float *__restrict__ scale,
                const float *__restrict__ base, mhc_params p, int64_t rows,
                float *__restrict__ pre_ws, float *__restrict__ post, float *__restrict__ comb,
                float *__restrict__ pre_out, float *__restrict__ mix_out) {
  const int64_t m = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (m >= rows) return;
  float dot[kPartial];
#pragma unroll
  for (int c = 0; c < kPartial; ++c) dot[c] = 0.f;
  for (int s = 0; s < kSlices; ++s) {
    const float *q = partials + ((int64_t)s * rows + m) * kPartial;
#pragma unroll
    for (int c = 0; c < kPartial; ++c) dot[c] += q[c];
  }
  const float rsq = 1.0f / sqrtf(dot[kMix] / (float)kK + p.rms_eps);
  float l[kMix];
#pragma unroll
  for (int c = 0; c < kMix; ++c) {
    const float mix = dot[c] * rsq;
    if (mix_out) mix_out[m * kMix + c] = mix;
    const int g = c < 4 ? 0 : (c < 8 ? 1 : 2);
    l[c] = fmaf(mix, __ldg(scale + g), __ldg(base + c));
  }
  float pr[kHC];
#pragma unroll
  for (int i = 0; i < kHC; ++i) {
    pr[i] = sigmoidf_(l[i]) + p.hc_pre_eps;
    post[m * kHC + i] = p.post_mult * sigmoidf_(l[4 + i]);
  }
  *reinterpret_cast<float4 *>(pre_ws + m * kHC) = make_float4(pr[0], pr[1], pr[2], pr[3]);
  if (pre_out) *reinterpret_cast<float4 *>(pre_out + m * kHC) = make_float4(pr[0], pr[1], pr[2], pr[3]);

  float C[kHC][kHC];
#pragma unroll
  for (int j = 0; j < kHC; ++j)
#pragma unroll
    for (int i = 0; i < kHC; ++i) C[j][i] = expf(l[8 + 4 * j + i]);
  const float eps = p.hc_sinkhorn_eps;
  for (int t = 0; t < p.sinkhorn_iters; ++t) {
#pragma unroll
    for (int j = 0; j < kHC; ++j) {
      const float d = ((C[j][0] + C[j][1]) + C[j][2]) + C[j][3] + eps;
#pragma unroll
      for (int i = 0; i < kHC; ++i) C[j][i] = C[j][i] / d;
    }
#pragma unroll
    for (int i = 0; i < kHC; ++i) {
      const float d = ((C[0][i] + C[1][i]) + C[2][i]) + C[3][i] + eps;
#pragma unroll
      for (int j = 0; j < kHC; ++j) C[j][i] = C[j][i] / d;
    }
  }
#pragma unroll
  for (int j = 0; j < kHC; ++j)
    *reinterpret_cast<float4 *>(comb + m * 16 + j * 4) = make_float4(C[j][0], C[j][1], C[j][2], C[j][3]);
}

// ---- combine (+ RMSNorm): one 128-thread block per row -----------------------
// kNorm: x_norm = bf16(y * rsqrt(mean y^2 + eps) * w) (the pre pass);
// otherwise y itself, cast once (hc_head: deepseek_v4.py, hc_head_torch).
constexpr int kCnThreads = 128;
constexpr int kCnChunks = kChunksPerStream / kCnThreads;   // 5
static_assert(kChunksPerStream % kCnThreads == 0, "");

// One row by one 128-thread block: y = sum_i pv_i R_i in fp32, then x_norm
// (kNorm) or y itself, cast once to bf16.
// kMx: the block also writes x_norm's MXFP8 codes (mxq, 8 per chunk) and
// linear block scales (mxs): a 32-column block is 4 consecutive chunks, held
// by 4 consecutive lanes.
template <bool kNorm, bool kMx = false>
__device__ __forceinline__ void combine_row(const uint4 *__restrict__ R, const float (&pv)[kHC],
                                            const uint4 *__restrict__ w, float norm_eps,
                                            uint4 *__restrict__ out, int64_t row,
                                            uint2 *__restrict__ mxq = nullptr,
                                            uint8_t *__restrict__ mxs = nullptr) {
  const int tid = threadIdx.x;
  const uint4 *r = R + row * (kHC * kChunksPerStream);

  float y[kCnChunks][8];
  float ss = 0.f;
#pragma unroll
  for (int q = 0; q < kCnChunks; ++q) {
    const int c = q * kCnThreads + tid;
    uint4 rv[kHC];
#pragma unroll
    for (int i = 0; i < kHC; ++i) rv[i] = ld_stream(r + i * kChunksPerStream + c);
    float rf[kHC][8];
#pragma unroll
    for (int i = 0; i < kHC; ++i) unpack8(rv[i], rf[i]);
#pragma unroll
    for (int e = 0; e < 8; ++e) {
      float a = pv[0] * rf[0][e];
#pragma unroll
      for (int i = 1; i < kHC; ++i) a = fmaf(pv[i], rf[i][e], a);
      y[q][e] = a;
      ss = fmaf(a, a, ss);
    }
  }
  uint4 *o = out + row * kChunksPerStream;
  if constexpr (!kNorm) {
#pragma unroll
    for (int q = 0; q < kCnChunks; ++q) st_stream(o + q * kCnThreads + tid, pack8_rn(y[q]));
    (void)w; (void)norm_eps; (void)ss;
  } else {
    __shared__ float red[kCnThreads / 32];
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, off);
    if ((tid & 31) == 0) red[tid >> 5] = ss;
    // the 4 combine warps only (a block may carry a Sinkhorn warp besides)
    asm volatile("bar.sync 1, %0;" ::"n"(kCnThreads) : "memory");
    const float tot = ((red[0] + red[1]) + red[2]) + red[3];
    const float rn = 1.0f / sqrtf(tot / (float)kH + norm_eps);

#pragma unroll
    for (int q = 0; q < kCnChunks; ++q) {
      const int c = q * kCnThreads + tid;
      float wf[8];
      unpack8(__ldg(w + c), wf);
      float v[8];
#pragma unroll
      for (int e = 0; e < 8; ++e) v[e] = (y[q][e] * rn) * wf[e];
      const uint4 xb = pack8_rn(v);
      st_stream(o + c, xb);
      if constexpr (kMx) {
        float vb[8];
        unpack8(xb, vb);                 // the bf16 values, as stored
        uint32_t sc;
        const uint2 codes = mx_block8(vb, sc);
        __stcs(mxq + row * kChunksPerStream + c, codes);
        if ((tid & 3) == 0) mxs[row * (kH / kMxBlock) + (c >> 2)] = (uint8_t)sc;
      }
    }
  }
}

// The row's 4x4 Sinkhorn (hc_split_sinkhorn) from its 16 comb logits, by one
// warp: lane e holds comb[e/4][e%4] (lanes 16..31 mirror 0..15); each
// iteration divides by the row sums (pairs (c0 + c1) + (c2 + c3)), then by
// the column sums, eps added to every sum.
__device__ __forceinline__ void sinkhorn_row(const float *__restrict__ logit,
                                             float *__restrict__ comb, int64_t row, float eps,
                                             int iters) {
  const int lane = threadIdx.x & 31, e = lane & 15;
  const unsigned full = 0xffffffffu;
  float cm = expf(__ldg(logit + row * 16 + e));
  for (int k = 0; k < iters; ++k) {
    float rs = cm + __shfl_xor_sync(full, cm, 1);
    rs = rs + __shfl_xor_sync(full, rs, 2);
    cm = cm / (rs + eps);
    float cs = cm + __shfl_xor_sync(full, cm, 4);
    cs = cs + __shfl_xor_sync(full, cs, 8);
    cm = cm / (cs + eps);
  }
  if (lane < 16) comb[row * 16 + e] = cm;
}

// kSink: a fifth warp runs the row's Sinkhorn while the four combine warps
// stream R (the stats launch leaves the comb logits in the workspace).
template <bool kNorm, bool kSink, bool kMx = false>
__global__ void __launch_bounds__(kCnThreads + 32)
combine_norm_kernel(const uint4 *__restrict__ R, const float4 *__restrict__ pre,
                    const uint4 *__restrict__ w, float norm_eps, uint4 *__restrict__ out,
                    const float *__restrict__ logit, float *__restrict__ comb, float sink_eps,
                    int iters, uint2 *__restrict__ mxq, uint8_t *__restrict__ mxs) {
  pdl_wait();
  pdl_trigger();
  // last rows first: after mhc_pre's stats launch the most recently read rows
  // are the ones still in L2
  const int64_t row = (int64_t)gridDim.x - 1 - blockIdx.x;
  if (threadIdx.x >= kCnThreads) {
    if constexpr (kSink) sinkhorn_row(logit, comb, row, sink_eps, iters);
    return;
  }
  const float4 pq = __ldg(pre + row);
  const float pv[kHC] = {pq.x, pq.y, pq.z, pq.w};
  combine_row<kNorm, kMx>(R, pv, w, norm_eps, out, row, mxq, mxs);
}

}  // namespace

size_t pre_simt_workspace_bytes(int64_t rows) {
  // partials [16][rows][25] fp32, then pre [rows][4] fp32 (256-byte aligned)
  size_t part = (size_t)kSlices * (size_t)rows * kPartial * sizeof(float);
  part = (part + 255) & ~(size_t)255;
  return part + (size_t)rows * kHC * sizeof(float);
}

cudaError_t launch_combine_norm(const uint16_t *R, const float *pre, const uint16_t *norm_w,
                                float norm_eps, int64_t rows, int64_t logical_rows,
                                uint16_t *x_norm, cudaStream_t s) {
  return launch_pdl(combine_norm_kernel<true, false>, dim3((unsigned)rows), dim3(kCnThreads), 0, s,
                    1, use_pdl(logical_rows), reinterpret_cast<const uint4 *>(R), reinterpret_cast<const float4 *>(pre),
                    reinterpret_cast<const uint4 *>(norm_w), norm_eps,
                    reinterpret_cast<uint4 *>(x_norm), nullptr, nullptr, 0.f, 0,
                    (uint2 *)nullptr, (uint8_t *)nullptr);
}

cudaError_t launch_combine_norm_sinkhorn(const uint16_t *R, const float *pre,
                                         const uint16_t *norm_w, float norm_eps,
                                         const float *logit, float *comb, float sink_eps,
                                         int iters, int64_t rows, int64_t logical_rows,
                                         uint16_t *x_norm, cudaStream_t s, uint8_t *mx_q,
                                         uint8_t *mx_s) {
  if (mx_q)
    return launch_pdl(combine_norm_kernel<true, true, true>, dim3((unsigned)rows),
                      dim3(kCnThreads + 32), 0, s, 1, use_pdl(logical_rows),
                      reinterpret_cast<const uint4 *>(R), reinterpret_cast<const float4 *>(pre),
                      reinterpret_cast<const uint4 *>(norm_w), norm_eps,
                      reinterpret_cast<uint4 *>(x_norm), logit, comb, sink_eps, iters,
                      reinterpret_cast<uint2 *>(mx_q), mx_s);
  return launch_pdl(combine_norm_kernel<true, true>, dim3((unsigned)rows), dim3(kCnThreads + 32),
                    0, s, 1, use_pdl(logical_rows), reinterpret_cast<const uint4 *>(R),
                    reinterpret_cast<const float4 *>(pre), reinterpret_cast<const uint4 *>(norm_w),
                    norm_eps, reinterpret_cast<uint4 *>(x_norm), logit, comb, sink_eps, iters,
                    (uint2 *)nullptr, (uint8_t *)nullptr);
}

cudaError_t launch_head_combine(const uint16_t *R, const float *pre, int64_t rows,
                                int64_t logical_rows, uint16_t *y, cudaStream_t s) {
  return launch_pdl(combine_norm_kernel<false, false>, dim3((unsigned)rows), dim3(kCnThreads), 0, s,
                    1, use_pdl(logical_rows), reinterpret_cast<const uint4 *>(R), reinterpret_cast<const float4 *>(pre),
                    nullptr, 0.f, reinterpret_cast<uint4 *>(y), nullptr, nullptr, 0.f, 0,
                    (uint2 *)nullptr, (uint8_t *)nullptr);
}

cudaError_t launch_pre_simt(const uint16_t *R, const float *fn, const float *scale,
                            const float *base, const uint16_t *norm_w, int64_t rows,
                            int64_t logical_rows, const mhc_params &p, void *workspace,
                            uint16_t *x_norm, float *post, float *comb, float *pre_out,
                            float *mix_out, cudaStream_t s) {
  float *partials = static_cast<float *>(workspace);
  size_t part = (size_t)kSlices * (size_t)rows * kPartial * sizeof(float);
  part = (part + 255) & ~(size_t)255;
  float *pre_ws = reinterpret_cast<float *>(static_cast<char *>(workspace) + part);

  dim3 g1((unsigned)((rows + kStatsRows - 1) / kStatsRows), kSlices);
  stats_partial_kernel<<<g1, kStatsThreads, 0, s>>>(R, fn, partials, rows);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  finalize_kernel<<<(unsigned)((rows + 127) / 128), 128, 0, s>>>(
      partials, scale, base, p, rows, pre_ws, post, comb, pre_out, mix_out);
  e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  return launch_combine_norm(R, pre_ws, norm_w, p.norm_eps, rows, logical_rows, x_norm, s);
}

}  // namespace mhc
