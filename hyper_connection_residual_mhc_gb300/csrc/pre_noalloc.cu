// pre_noalloc.cu -- the scratch of the allocation-free mhc_pre variant.
//
// Some callers cannot hand this library device scratch: a framework whose
// caching allocator has reserved the device memory for itself, a plugin or
// operator interface whose enqueue function must not allocate, a latency-
// critical serving loop that cannot afford cudaMalloc/cudaFree (which may
// synchronise the device), or a plain C / FFI caller with no device allocator
// at hand.  For them mhc_pre_noalloc runs the CUDA-core pre path with its
// scratch in the fixed array below instead of a caller workspace.
//
// The array lives in every GPU that loads the library, until the process
// exits: kNoAllocMaxRows rows' worth (about 25.3 MiB).  Its name is only a
// host-side stand-in in host code; the device address is looked up once per
// device with cudaGetSymbolAddress, with that device current, on the first
// call made on that device, and cached.
#include <mutex>

#include "mhc_common.cuh"

namespace mhc {

constexpr int64_t kNoAllocMaxRows = 16384;

// Same layout launch_pre_simt uses: partials [16][rows][25] fp32 padded to
// 256 bytes, then pre [rows][4] fp32.
constexpr size_t kNoAllocPartialBytes =
    ((size_t)16 * kNoAllocMaxRows * 25 * sizeof(float) + 255) / 256 * 256;
constexpr size_t kNoAllocBytes = kNoAllocPartialBytes + (size_t)kNoAllocMaxRows * 4 * sizeof(float);

static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocBytes];

namespace {
constexpr int kMaxDevices = 64;
std::mutex g_noalloc_mu;
void *g_noalloc_ptr[kMaxDevices] = {};
}  // namespace

int64_t noalloc_max_rows() { return kNoAllocMaxRows; }

// Device address of the scratch array on the current device (looked up once
// per device, with that device current).
static cudaError_t noalloc_scratch(void **out) {
  int dev = -1;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lock(g_noalloc_mu);
  if (!g_noalloc_ptr[dev]) {
    void *p = nullptr;
    e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
    if (e != cudaSuccess) return e;
    g_noalloc_ptr[dev] = p;
  }
  *out = g_noalloc_ptr[dev];
  return cudaSuccess;
}

cudaError_t launch_pre_noalloc(const uint16_t *R, const float *fn, const float *scale,
                               const float *base, const uint16_t *norm_w, int64_t rows,
                               int64_t logical_rows, const mhc_params &p, uint16_t *x_norm,
                               float *post, float *comb, float *pre_out, float *mix_out,
                               cudaStream_t s) {
  // Every word of scratch this path reads is written earlier in the same
  // call (each partial slot by stats_partial, each pre by finalize), so the
  // previous call's leftovers need no clearing.
  if (rows > kNoAllocMaxRows || pre_simt_workspace_bytes(rows) > kNoAllocBytes)
    return cudaErrorInvalidValue;
  void *scratch = nullptr;
  cudaError_t e = noalloc_scratch(&scratch);
  if (e != cudaSuccess) return e;
  return launch_pre_simt(R, fn, scale, base, norm_w, rows, logical_rows, p, scratch, x_norm,
                         post, comb, pre_out, mix_out, s);
}

}  // namespace mhc
