// mxfp8.cu -- MXFP8 output of bf16 rows and the 128x4 scale layout
// (prefill_sp.py, _mxfp8_quantize and swizzle_128x4: the attention input is
// quantized per row and per 32 columns to E4M3 codes with ue8m0 scales, and
// the linear scales are then tiled 128x4 for the GEMM that reads them).
//
// On the prefill path mhc_pre's combine kernel writes the codes itself, from
// the x_norm values it has in registers (mx_block8 in mhc_common.cuh).  The
// kernels here serve everything else: decode-size chunks (whose one-launch
// kernel writes bf16 x_norm only), any bf16 rows a caller has, and the
// scale tiling.  Both are HBM-streaming: the quantizer reads 2 bytes and
// writes 1 + 1/32 bytes per value; the tiling moves 1 byte per scale.
#include "mhc_common.cuh"

namespace mhc {
namespace {

constexpr int kMxThreads = 256;

// One 16-byte chunk (8 values) per lane, warp-uniform trip count so that the
// 4-lane block reductions in mx_block8 always see a full warp.  chunks is a
// multiple of 4 (cols % 32 == 0), so a lane group is all valid or all not.
__global__ void __launch_bounds__(kMxThreads)
mx_quantize_kernel(const uint4 *__restrict__ x, int64_t chunks, uint2 *__restrict__ q,
                   uint8_t *__restrict__ s) {
  pdl_wait();
  pdl_trigger();
  const int lane = threadIdx.x & 31;
  const int64_t warp = (int64_t)blockIdx.x * (kMxThreads / 32) + (threadIdx.x >> 5);
  const int64_t step = (int64_t)gridDim.x * kMxThreads;
  for (int64_t c0 = warp * 32; c0 < chunks; c0 += step) {
    const int64_t c = c0 + lane;
    const bool ok = c < chunks;
    float v[8];
    unpack8(ok ? ld_stream(x + c) : make_uint4(0u, 0u, 0u, 0u), v);
    uint32_t sc;
    const uint2 codes = mx_block8(v, sc);
    if (ok) {
      __stcs(q + c, codes);
      if ((lane & 3) == 0) s[c >> 2] = (uint8_t)sc;
    }
  }
}

// One 4-byte word of the tiled layout per thread: a word is the 4 scales of
// one row's 4-group tile, so it is also one aligned word of the linear
// layout.  Word p of tile t = p / 128 (tile (tm, tg), row-tile-major) holds
// row tm*128 + ((p % 128) % 4)*32 + (p % 128) / 4, groups 4*tg .. 4*tg + 3.
__global__ void __launch_bounds__(kMxThreads)
mx_swizzle_kernel(const uint32_t *__restrict__ s, int64_t rows, int64_t groups4,
                  uint32_t *__restrict__ out, int64_t words) {
  pdl_wait();
  pdl_trigger();
  const int64_t step = (int64_t)gridDim.x * kMxThreads;
  for (int64_t p = (int64_t)blockIdx.x * kMxThreads + threadIdx.x; p < words; p += step) {
    const int64_t t = p >> 7;
    const int in = (int)(p & 127);
    const int64_t tm = t / groups4, tg = t % groups4;
    const int64_t m = tm * 128 + (in & 3) * 32 + (in >> 2);
    out[p] = m < rows ? __ldg(s + m * groups4 + tg) : 0u;
  }
}

inline unsigned stream_grid(int64_t work) {
  // at most 8 resident 256-thread blocks on each of the 152 SMs; grid-stride beyond
  const int64_t cap = 152 * 8;
  const int64_t g = (work + kMxThreads - 1) / kMxThreads;
  return (unsigned)(g < 1 ? 1 : (g > cap ? cap : g));
}

}  // namespace

cudaError_t launch_mx_quantize(const uint16_t *x, int64_t rows, int64_t cols,
                               int64_t logical_rows, uint8_t *q, uint8_t *s, cudaStream_t st) {
  const int64_t chunks = rows * cols / kChunk;
  // whole warps: the grid covers chunks rounded up to 32 lanes
  return launch_pdl(mx_quantize_kernel, dim3(stream_grid((chunks + 31) / 32 * 32)),
                    dim3(kMxThreads), 0, st, 1, use_pdl(logical_rows),
                    reinterpret_cast<const uint4 *>(x), chunks, reinterpret_cast<uint2 *>(q), s);
}

cudaError_t launch_mx_swizzle(const uint8_t *s, int64_t rows, int64_t groups, uint8_t *out,
                              cudaStream_t st) {
  const int64_t words = (rows + 127) / 128 * 128 * (groups / 4);
  return launch_pdl(mx_swizzle_kernel, dim3(stream_grid(words)), dim3(kMxThreads), 0, st, 1,
                    use_pdl(rows), reinterpret_cast<const uint32_t *>(s), rows, groups / 4,
                    reinterpret_cast<uint32_t *>(out), words);
}

}  // namespace mhc
