// pre_simt.cu -- the streaming combine + RMSNorm launches: one 128-thread
// block per row computes y = sum_i pre_i R_i in fp32, then x_norm, rounded
// once to bf16 (deepseek_v4.py, DeepseekV4DecoderLayer.hc_pre: the combine;
// RMSNorm fused as in prefill_sp.py, hc_combine_norm_rows).  Used by
// mhc_combine_norm, and by mhc_fused_post_pre after its tensor-core launch,
// which also hands a fifth warp per row the comb logits for the Sinkhorn.
//
// Every row is reduced in one fixed order that depends on nothing but the
// row's own data: per-thread strides and the tree of the block reductions are
// compile-time constants.  Row ranges therefore give the whole-chunk bits.
#include "mhc_common.cuh"

namespace mhc {
namespace {

// ---- combine + RMSNorm: one 128-thread block per row --------------------------
// x_norm = bf16(y * rsqrt(mean y^2 + eps) * w)
constexpr int kCnThreads = 128;
constexpr int kCnChunks = kChunksPerStream / kCnThreads;   // 5
static_assert(kChunksPerStream % kCnThreads == 0, "");

// One row by one 128-thread block: y = sum_i pv_i R_i in fp32, then x_norm,
// cast once to bf16.
// kMx: the block also writes x_norm's MXFP8 codes (mxq, 8 per chunk) and
// linear block scales (mxs): a 32-column block is 4 consecutive chunks, held
// by 4 consecutive lanes.
template <bool kMx = false>
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
  {
    __shared__ float red[kCnThreads / 32];
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, off);
    if ((tid & 31) == 0) red[tid >> 5] = ss;
    // the 4 combine warps only (a block may carry a Sinkhorn warp besides)
    asm volatile("bar.sync 1, %0;" ::"n"(kCnThreads) : "memory");
    const float tot = ((red[0] + red[1]) + red[2]) + red[3];
    const float rn = rsqrt_nr(fmaf(tot, 1.0f / (float)kH, norm_eps));

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
// iteration scales by the reciprocals of the row sums (pairs (c0 + c1) +
// (c2 + c3)), then of the column sums, eps added to every sum.
__device__ __forceinline__ void sinkhorn_row(const float *__restrict__ logit,
                                             float *__restrict__ comb, int64_t row, float eps,
                                             int iters) {
  const int lane = threadIdx.x & 31, e = lane & 15;
  const unsigned full = 0xffffffffu;
  float cm = expf(__ldg(logit + row * 16 + e));
  for (int k = 0; k < iters; ++k) {
    float rs = cm + __shfl_xor_sync(full, cm, 1);
    rs = rs + __shfl_xor_sync(full, rs, 2);
    cm = cm * rcp_nr(rs + eps);
    float cs = cm + __shfl_xor_sync(full, cm, 4);
    cs = cs + __shfl_xor_sync(full, cs, 8);
    cm = cm * rcp_nr(cs + eps);
  }
  if (lane < 16) comb[row * 16 + e] = cm;
}

// kSink: a fifth warp runs the row's Sinkhorn while the four combine warps
// stream R (the fused call's tensor-core launch leaves the comb logits in the
// workspace).
template <bool kSink, bool kMx = false>
__global__ void __launch_bounds__(kCnThreads + 32)
combine_norm_kernel(const uint4 *__restrict__ R, const float4 *__restrict__ pre,
                    const uint4 *__restrict__ w, float norm_eps, uint4 *__restrict__ out,
                    const float *__restrict__ logit, float *__restrict__ comb, float sink_eps,
                    int iters, uint2 *__restrict__ mxq, uint8_t *__restrict__ mxs) {
  pdl_wait();
  pdl_trigger();
  // last rows first: after the fused call's tensor-core launch the most
  // recently written rows are the ones still in L2
  const int64_t row = (int64_t)gridDim.x - 1 - blockIdx.x;
  if (threadIdx.x >= kCnThreads) {
    if constexpr (kSink) sinkhorn_row(logit, comb, row, sink_eps, iters);
    return;
  }
  const float4 pq = __ldg(pre + row);
  const float pv[kHC] = {pq.x, pq.y, pq.z, pq.w};
  combine_row<kMx>(R, pv, w, norm_eps, out, row, mxq, mxs);
}

}  // namespace

cudaError_t launch_combine_norm(const uint16_t *R, const float *pre, const uint16_t *norm_w,
                                float norm_eps, int64_t rows, int64_t logical_rows,
                                uint16_t *x_norm, cudaStream_t s) {
  return launch_pdl(combine_norm_kernel<false>, dim3((unsigned)rows), dim3(kCnThreads), 0, s,
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
    return launch_pdl(combine_norm_kernel<true, true>, dim3((unsigned)rows),
                      dim3(kCnThreads + 32), 0, s, 1, use_pdl(logical_rows),
                      reinterpret_cast<const uint4 *>(R), reinterpret_cast<const float4 *>(pre),
                      reinterpret_cast<const uint4 *>(norm_w), norm_eps,
                      reinterpret_cast<uint4 *>(x_norm), logit, comb, sink_eps, iters,
                      reinterpret_cast<uint2 *>(mx_q), mx_s);
  return launch_pdl(combine_norm_kernel<true>, dim3((unsigned)rows), dim3(kCnThreads + 32),
                    0, s, 1, use_pdl(logical_rows), reinterpret_cast<const uint4 *>(R),
                    reinterpret_cast<const float4 *>(pre), reinterpret_cast<const uint4 *>(norm_w),
                    norm_eps, reinterpret_cast<uint4 *>(x_norm), logit, comb, sink_eps, iters,
                    (uint2 *)nullptr, (uint8_t *)nullptr);
}

}  // namespace mhc
