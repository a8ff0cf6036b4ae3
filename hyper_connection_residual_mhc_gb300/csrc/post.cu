// post.cu -- hc_post: R_out[m, i, h] = post[m, i] * y[m, h] + sum_j comb[m, j, i] * R[m, j, h]
// (deepseek_v4.py, DeepseekV4DecoderLayer.hc_post, hc_post_torch_impl), fp32
// arithmetic, one rounding to bf16.
//
// Pure streaming: per row it reads 40960 B of R and 10240 B of y and writes
// 40960 B.  One thread owns one 8-column chunk of one row across all four
// streams: five independent 16-byte loads in flight, 32 fp32 FMA chains, four
// 16-byte stores; a block is 64 threads.  post/comb (80 B per row) come through L1.  The arithmetic of
// an element depends only on that element's inputs, so any row range gives the
// whole-chunk bits.
#include "mhc_common.cuh"

namespace mhc {
namespace {

// 64-thread blocks: at 64 registers a thread an SM holds 1024 threads whatever
// the block size, and finer blocks stream faster (M = 16384: 0.2191 ms against
// 0.2212 / 0.2254 / 0.2318 ms with 128 / 256 / 512 threads; 32 threads,
// 0.3335 ms, run out of blocks an SM)
constexpr int kPostThreads = 64;

__global__ void __launch_bounds__(kPostThreads)
post_kernel(const uint4 *__restrict__ R, const uint4 *__restrict__ y,
            const float4 *__restrict__ post, const float4 *__restrict__ comb,
            uint4 *__restrict__ out, int64_t n_chunks) {
  pdl_wait();
  pdl_trigger();
  const int64_t t = (int64_t)blockIdx.x * kPostThreads + threadIdx.x;
  if (t >= n_chunks) return;
  const int64_t row = t / kChunksPerStream;
  const int c = (int)(t - row * kChunksPerStream);

  const uint4 *r = R + row * (kHC * kChunksPerStream) + c;
  uint4 rv[kHC];
#pragma unroll
  for (int j = 0; j < kHC; ++j) rv[j] = ld_stream(r + j * kChunksPerStream);
  const uint4 yv = ld_stream(y + row * kChunksPerStream + c);

  const float4 pw = __ldg(post + row);
  float cb[kHC][kHC];  // cb[j][i]
#pragma unroll
  for (int j = 0; j < kHC; ++j) {
    const float4 q = __ldg(comb + row * kHC + j);
    cb[j][0] = q.x; cb[j][1] = q.y; cb[j][2] = q.z; cb[j][3] = q.w;
  }
  const float pv[kHC] = {pw.x, pw.y, pw.z, pw.w};

  uint4 ov[kHC];
  post_chunk(rv, yv, pv, cb, ov);
  uint4 *o = out + row * (kHC * kChunksPerStream) + c;
#pragma unroll
  for (int i = 0; i < kHC; ++i) st_stream(o + i * kChunksPerStream, ov[i]);
}

}  // namespace

cudaError_t launch_post(const uint16_t *R, const uint16_t *y, const float *post,
                        const float *comb, int64_t rows, int64_t logical_rows,
                        uint16_t *R_out, cudaStream_t s) {
  const int64_t n_chunks = rows * kChunksPerStream;
  const int64_t blocks = (n_chunks + kPostThreads - 1) / kPostThreads;
  return launch_pdl(post_kernel, dim3((unsigned)blocks), dim3(kPostThreads), 0, s, 1,
                    use_pdl(logical_rows),
                    reinterpret_cast<const uint4 *>(R), reinterpret_cast<const uint4 *>(y),
                    reinterpret_cast<const float4 *>(post), reinterpret_cast<const float4 *>(comb),
                    reinterpret_cast<uint4 *>(R_out), n_chunks);
}

}  // namespace mhc
