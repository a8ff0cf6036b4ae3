// abi.cu -- the extern "C" entry points of libmhc: host-side validation, then
// the internal launchers.  Nothing here allocates device memory.
#include <atomic>
#include <cmath>
#include <cstring>
#include <string>

#include "mhc_common.cuh"

namespace {

thread_local std::string g_last_cuda_error;

int cuda_fail(cudaError_t e) {
  g_last_cuda_error = std::string(cudaGetErrorName(e)) + ": " + cudaGetErrorString(e);
  return MHC_ERR_CUDA;
}

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

bool finite_nonneg(float v) { return std::isfinite(v) && v >= 0.f; }

struct Span {
  uintptr_t lo, hi;
};
Span span(const void *p, size_t bytes) {
  uintptr_t a = reinterpret_cast<uintptr_t>(p);
  return {a, a + bytes};
}
bool overlap(Span a, Span b) { return a.lo < b.hi && b.lo < a.hi; }

// rows are indexed with 32-bit block counts in places: keep rows * 640 chunks
// (the largest per-row grid) inside a signed 32-bit grid dimension times 256.
constexpr int64_t kMaxRows = (int64_t)1 << 24;
// columns of a row the MXFP8 quantizer takes: a 16M-row by 64k-column call
// stays below 2^40 values, well inside the kernels' 64-bit chunk indices
constexpr int64_t kMaxMxCols = (int64_t)1 << 16;

int check_rows(int64_t rows, int64_t logical_rows) {
  if (rows < 0 || logical_rows < rows || rows > kMaxRows) return MHC_ERR_SHAPE;
  return MHC_OK;
}

// The kernels are built for sm_103a only.  Check the current device once per
// device (cached), after argument validation, before the first launch.
int check_device() {
  int dev = -1;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_fail(e);
  // bit d set: device d verified (callers may come from several host threads)
  static std::atomic<unsigned> ok_mask{0u};
  if (dev >= 0 && dev < 32 && (ok_mask.load(std::memory_order_relaxed) >> dev) & 1u)
    return MHC_OK;
  int major = 0, minor = 0;
  e = cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev);
  if (e == cudaSuccess) e = cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev);
  if (e != cudaSuccess) return cuda_fail(e);
  if (major != 10 || minor != 3) return MHC_ERR_DEVICE;
  if (dev >= 0 && dev < 32) ok_mask.fetch_or(1u << dev, std::memory_order_relaxed);
  return MHC_OK;
}

}  // namespace

extern "C" {

void mhc_default_params(mhc_params *p) {
  if (!p) return;
  p->rms_eps = 1e-6f;
  p->hc_pre_eps = 1e-6f;
  p->hc_sinkhorn_eps = 1e-6f;
  p->norm_eps = 1e-6f;
  p->post_mult = 2.0f;
  p->sinkhorn_iters = 20;
}

const char *mhc_strerror(int code) {
  switch (code) {
    case MHC_OK: return "ok";
    case MHC_ERR_NULL: return "a required pointer is NULL";
    case MHC_ERR_SHAPE:
      return "bad shape (rows < 0, logical_rows < rows, too many rows, or a bad column or "
             "group count)";
    case MHC_ERR_ALIGN: return "a tensor pointer is not 16-byte aligned";
    case MHC_ERR_PARAM: return "bad scalar parameter (eps < 0 or not finite, iterations < 1)";
    case MHC_ERR_OVERLAP: return "an output buffer overlaps an input buffer";
    case MHC_ERR_WORKSPACE: return "workspace missing, misaligned or too small";
    case MHC_ERR_CUDA: return "a CUDA call failed";
    case MHC_ERR_DEVICE: return "the current device is not an sm_103 GPU";
    case MHC_ERR_SCRATCH_LIMIT:
      return "rows exceed a fixed scratch size (not returned by this build)";
    case MHC_ERR_ALLOC: return "a device allocation failed (mhc_prepare_weights)";
    default: return "unknown libmhc error code";
  }
}

const char *mhc_last_cuda_error(void) { return g_last_cuda_error.c_str(); }

namespace {
size_t gate_bytes(int64_t rows) {
  return ((size_t)rows * MHC_HC * sizeof(float) + 255) & ~(size_t)255;
}
size_t logit_bytes(int64_t rows) {
  return ((size_t)rows * 16 * sizeof(float) + 255) & ~(size_t)255;
}
}  // namespace

size_t mhc_pre_workspace_bytes(int64_t rows) {
  if (rows <= 0) return 0;
  // mhc_pre: fn's operand image for the streamed one-pass build (chunks of
  // kStreamMinRows rows and more).  The fused call's tensor-core launch hands
  // its combine launch the pre gates [rows, 4] fp32, then the comb logits
  // [rows, 16] fp32, each 256-byte rounded.  mhc_hc_head and the decode-size
  // paths use none of it.
  const size_t handoff = gate_bytes(rows) + logit_bytes(rows);
  const size_t img = mhc::fn_b_img_bytes();
  return handoff > img ? handoff : img;
}

size_t mhc_fused_post_pre_workspace_bytes(int64_t rows) {
  if (rows <= 0) return 0;
  // what mhc_pre's launches hand each other, then fn in the fused kernel's
  // B-operand image (written by the call itself)
  return mhc_pre_workspace_bytes(rows) + mhc::fused_fn_bytes();
}

int mhc_kernel_status_detail(uint32_t *where64) {
  if (!where64) return MHC_ERR_NULL;
  cudaError_t e = mhc::onepass_error_where(where64);
  return e == cudaSuccess ? MHC_OK : cuda_fail(e);
}

int mhc_kernel_status(uint32_t *status, int reset) {
  if (!status) return MHC_ERR_NULL;
  unsigned int w = 0, w2 = 0, w3 = 0, w4 = 0, w5 = 0;
  cudaError_t e = mhc::head_tile_error_word(&w, reset != 0);
  if (e == cudaSuccess) e = mhc::fused_post_pre_error_word(&w2, reset != 0);
  if (e == cudaSuccess) e = mhc::head_error_word(&w3, reset != 0);
  if (e == cudaSuccess) e = mhc::onepass_error_word(&w4, reset != 0);
  if (e == cudaSuccess) e = mhc::decode_error_word(&w5, reset != 0);
  if (e != cudaSuccess) return cuda_fail(e);
  *status = w | w2 | w3 | w4 | w5;
  return MHC_OK;
}

namespace {
// mhc_pre, mhc_pre_prepared and mhc_pre_mxfp8: fn is the fp32 weight (the
// caller's, or the handle's copy); fn_b_img is NULL or the handle's image of
// fn's operand tiles; mx_q / mx_s are NULL or x_norm's MXFP8 codes and linear
// scales
int pre_impl(const uint16_t *R, const float *fn, const uint8_t *fn_b_img, const float *scale,
             const float *base, const uint16_t *norm_w, int64_t rows, int64_t logical_rows,
             const mhc_params *p_in, void *workspace, size_t workspace_bytes, uint16_t *x_norm,
             float *post, float *comb, float *pre_out, float *mix_out, void *stream,
             uint8_t *mx_q = nullptr, uint8_t *mx_s = nullptr, bool ws_required = true) {
  mhc_params p;
  if (p_in) p = *p_in; else mhc_default_params(&p);
  if (int e = check_rows(rows, logical_rows)) return e;
  if (!finite_nonneg(p.rms_eps) || !finite_nonneg(p.hc_pre_eps) ||
      !finite_nonneg(p.hc_sinkhorn_eps) || !finite_nonneg(p.norm_eps) ||
      !std::isfinite(p.post_mult) || p.sinkhorn_iters < 1 || p.sinkhorn_iters > 100000)
    return MHC_ERR_PARAM;
  if (rows == 0) return MHC_OK;
  if (!R || !fn || !scale || !base || !norm_w || !x_norm || !post || !comb) return MHC_ERR_NULL;
  const void *al[] = {R, fn, scale, base, norm_w, x_norm, post, comb};
  for (const void *q : al)
    if (!aligned16(q)) return MHC_ERR_ALIGN;
  if ((pre_out && !aligned16(pre_out)) || (mix_out && !aligned16(mix_out))) return MHC_ERR_ALIGN;
  if ((mx_q == nullptr) != (mx_s == nullptr)) return MHC_ERR_NULL;
  if (mx_q && (!aligned16(mx_q) || !aligned16(mx_s))) return MHC_ERR_ALIGN;
  const size_t need = ws_required ? mhc_pre_workspace_bytes(rows) : 0;
  if (need > 0 && (!workspace || workspace_bytes < need ||
                   (reinterpret_cast<uintptr_t>(workspace) & 255u)))
    return MHC_ERR_WORKSPACE;

  const size_t nr = (size_t)rows;
  const Span ins[] = {span(R, nr * MHC_K * 2), span(fn, (size_t)MHC_MIX * MHC_K * 4),
                      span(scale, 12), span(base, MHC_MIX * 4), span(norm_w, MHC_HIDDEN * 2)};
  Span outs[8];
  int n_out = 0;
  outs[n_out++] = span(x_norm, nr * MHC_HIDDEN * 2);
  if (mx_q) {
    outs[n_out++] = span(mx_q, nr * MHC_HIDDEN);
    outs[n_out++] = span(mx_s, nr * (MHC_HIDDEN / 32));
  }
  outs[n_out++] = span(post, nr * MHC_HC * 4);
  outs[n_out++] = span(comb, nr * MHC_HC * MHC_HC * 4);
  if (pre_out) outs[n_out++] = span(pre_out, nr * MHC_HC * 4);
  if (mix_out) outs[n_out++] = span(mix_out, nr * MHC_MIX * 4);
  if (need) outs[n_out++] = span(workspace, need);
  for (int a = 0; a < n_out; ++a) {
    for (const Span &b : ins)
      if (overlap(outs[a], b)) return MHC_ERR_OVERLAP;
    for (int b = a + 1; b < n_out; ++b)
      if (overlap(outs[a], outs[b])) return MHC_ERR_OVERLAP;
  }

  if (int e = check_device()) return e;
  const cudaStream_t s = static_cast<cudaStream_t>(stream);
  cudaError_t ce;
  if (logical_rows <= mhc::kDecodeMaxRows) {
    // decode-size chunk: latency-shaped CUDA-core path (keyed on the chunk's
    // row count, so every shard of the chunk takes it)
    ce = mhc::launch_pre_decode(R, fn, scale, base, norm_w, rows, logical_rows, p, x_norm, post,
                                comb, pre_out, mix_out, s, /*fn_stable=*/fn_b_img != nullptr);
    // the decode kernel writes bf16 x_norm only; its MXFP8 follows in a
    // second, streaming launch
    if (ce == cudaSuccess && mx_q)
      ce = mhc::launch_mx_quantize(x_norm, rows, MHC_HIDDEN, logical_rows, mx_q, mx_s, s);
  } else {
    // one launch that reads R from HBM once (fn's operand tiles from the
    // handle's image when prepared).  A chunk that takes the streamed build
    // without a handle gets its image written into the workspace first, so
    // mhc_pre and mhc_pre_prepared give the same bits; without a workspace
    // (mhc_pre_noalloc) the resident build runs.
    const uint8_t *img = fn_b_img;
    ce = cudaSuccess;
    if (!img && logical_rows >= mhc::kStreamMinRows && workspace &&
        workspace_bytes >= mhc::fn_b_img_bytes()) {
      uint8_t *ws_img = static_cast<uint8_t *>(workspace);
      ce = mhc::launch_fn_b_img(fn, ws_img, s);
      img = ws_img;
    }
    if (ce == cudaSuccess)
      ce = mhc::launch_pre_onepass(R, fn, img, scale, base, norm_w, rows, logical_rows, p,
                                   x_norm, post, comb, pre_out, mix_out, s, mx_q, mx_s);
  }
  return ce == cudaSuccess ? MHC_OK : cuda_fail(ce);
}
}  // namespace

int mhc_pre(const uint16_t *R, const float *fn, const float *scale, const float *base,
            const uint16_t *norm_w, int64_t rows, int64_t logical_rows, const mhc_params *p,
            void *workspace, size_t workspace_bytes, uint16_t *x_norm, float *post,
            float *comb, float *pre_out, float *mix_out, void *stream) {
  return pre_impl(R, fn, nullptr, scale, base, norm_w, rows, logical_rows, p, workspace,
                  workspace_bytes, x_norm, post, comb, pre_out, mix_out, stream);
}

// ---- prepared weights --------------------------------------------------------------
struct mhc_weights {
  int device;
  float *fn32;      // device copy of fn [24, 20480] fp32 (decode paths)
  uint8_t *img;     // the one-pass pre kernel's bf16 hi/lo operand tiles of fn, all 16 ranks
  uint8_t *img64;   // the fused post -> pre kernel's image (64-byte swizzled 32-k blocks)
};

int mhc_prepare_weights(const float *fn, mhc_weights **out, void *stream) {
  if (!fn || !out) return MHC_ERR_NULL;
  *out = nullptr;
  if (!aligned16(fn)) return MHC_ERR_ALIGN;
  if (int e = check_device()) return e;
  int dev = 0;
  cudaError_t ce = cudaGetDevice(&dev);
  if (ce != cudaSuccess) return cuda_fail(ce);
  const size_t fn_bytes = (size_t)MHC_MIX * MHC_K * sizeof(float);
  mhc_weights *w = new mhc_weights{dev, nullptr, nullptr, nullptr};
  auto drop = [&]() {
    cudaFree(w->fn32);
    cudaFree(w->img);
    cudaFree(w->img64);
    delete w;
  };
  ce = cudaMalloc(reinterpret_cast<void **>(&w->fn32), fn_bytes);
  if (ce == cudaSuccess)
    ce = cudaMalloc(reinterpret_cast<void **>(&w->img), mhc::fn_b_img_bytes());
  if (ce == cudaSuccess)
    ce = cudaMalloc(reinterpret_cast<void **>(&w->img64), mhc::fused_fn_bytes());
  if (ce != cudaSuccess) {
    drop();
    cuda_fail(ce);
    return MHC_ERR_ALLOC;
  }
  const cudaStream_t s = static_cast<cudaStream_t>(stream);
  ce = cudaMemcpyAsync(w->fn32, fn, fn_bytes, cudaMemcpyDeviceToDevice, s);
  if (ce == cudaSuccess) ce = mhc::launch_fn_b_img(fn, w->img, s);
  if (ce == cudaSuccess) ce = mhc::launch_fn_prep_sw64(fn, w->img64, s, false);
  if (ce != cudaSuccess) {
    drop();
    return cuda_fail(ce);
  }
  *out = w;
  return MHC_OK;
}

int mhc_release_weights(mhc_weights *w) {
  if (!w) return MHC_OK;
  cudaError_t e1 = cudaFree(w->fn32), e2 = cudaFree(w->img), e3 = cudaFree(w->img64);
  delete w;
  if (e1 != cudaSuccess) return cuda_fail(e1);
  if (e2 != cudaSuccess) return cuda_fail(e2);
  if (e3 != cudaSuccess) return cuda_fail(e3);
  return MHC_OK;
}

int mhc_pre_prepared(const uint16_t *R, const mhc_weights *w, const float *scale,
                     const float *base, const uint16_t *norm_w, int64_t rows,
                     int64_t logical_rows, const mhc_params *p, void *workspace,
                     size_t workspace_bytes, uint16_t *x_norm, float *post, float *comb,
                     float *pre_out, float *mix_out, void *stream) {
  if (!w) return MHC_ERR_NULL;
  int dev = -1;
  if (cudaGetDevice(&dev) == cudaSuccess && dev != w->device) return MHC_ERR_DEVICE;
  return pre_impl(R, w->fn32, w->img, scale, base, norm_w, rows, logical_rows, p, workspace,
                  workspace_bytes, x_norm, post, comb, pre_out, mix_out, stream);
}

int mhc_pre_mxfp8(const uint16_t *R, const mhc_weights *w, const float *scale, const float *base,
                  const uint16_t *norm_w, int64_t rows, int64_t logical_rows,
                  const mhc_params *p, void *workspace, size_t workspace_bytes,
                  uint16_t *x_norm, uint8_t *x_q, uint8_t *x_s, float *post, float *comb,
                  void *stream) {
  if (!w) return MHC_ERR_NULL;
  if (rows > 0 && (!x_q || !x_s)) return MHC_ERR_NULL;
  int dev = -1;
  if (cudaGetDevice(&dev) == cudaSuccess && dev != w->device) return MHC_ERR_DEVICE;
  return pre_impl(R, w->fn32, w->img, scale, base, norm_w, rows, logical_rows, p, workspace,
                  workspace_bytes, x_norm, post, comb, nullptr, nullptr, stream, x_q, x_s);
}

int mhc_quantize_mxfp8(const uint16_t *x, int64_t rows, int64_t cols, int64_t logical_rows,
                       uint8_t *q, uint8_t *s, void *stream) {
  if (int e = check_rows(rows, logical_rows)) return e;
  if (cols <= 0 || cols % 32 != 0 || cols > kMaxMxCols) return MHC_ERR_SHAPE;
  if (rows == 0) return MHC_OK;
  if (!x || !q || !s) return MHC_ERR_NULL;
  if (!aligned16(x) || !aligned16(q) || !aligned16(s)) return MHC_ERR_ALIGN;
  const size_t n = (size_t)rows * (size_t)cols;
  const Span sp[] = {span(x, n * 2), span(q, n), span(s, n / 32)};
  for (int a = 0; a < 3; ++a)
    for (int b = a + 1; b < 3; ++b)
      if (overlap(sp[a], sp[b])) return MHC_ERR_OVERLAP;
  if (int e = check_device()) return e;
  cudaError_t ce = mhc::launch_mx_quantize(x, rows, cols, logical_rows, q, s,
                                           static_cast<cudaStream_t>(stream));
  return ce == cudaSuccess ? MHC_OK : cuda_fail(ce);
}

size_t mhc_swizzle_scales_128x4_bytes(int64_t rows, int64_t groups) {
  if (rows <= 0 || groups <= 0 || rows > kMaxRows || groups > kMaxMxCols / 32) return 0;
  return (size_t)((rows + 127) / 128 * 128) * (size_t)groups;
}

int mhc_swizzle_scales_128x4(const uint8_t *s, int64_t rows, int64_t groups, uint8_t *out,
                             void *stream) {
  if (rows < 0 || rows > kMaxRows) return MHC_ERR_SHAPE;
  if (groups <= 0 || groups % 4 != 0 || groups > kMaxMxCols / 32) return MHC_ERR_SHAPE;
  if (rows == 0) return MHC_OK;
  if (!s || !out) return MHC_ERR_NULL;
  if (!aligned16(s) || !aligned16(out)) return MHC_ERR_ALIGN;
  if (overlap(span(s, (size_t)rows * (size_t)groups),
              span(out, mhc_swizzle_scales_128x4_bytes(rows, groups))))
    return MHC_ERR_OVERLAP;
  if (int e = check_device()) return e;
  cudaError_t ce = mhc::launch_mx_swizzle(s, rows, groups, out, static_cast<cudaStream_t>(stream));
  return ce == cudaSuccess ? MHC_OK : cuda_fail(ce);
}

int64_t mhc_pre_noalloc_max_rows(void) { return kMaxRows; }

// Allocation-free mhc_pre: mhc_pre's kernels (the decode-size launch and the
// one-pass launch) take no scratch, so this is mhc_pre without the workspace
// argument.  Below kStreamMinRows logical rows it runs mhc_pre's launches and
// gives its bits; from there on, with no room for fn's image, the one-pass
// launch keeps fn's tiles resident (16-CTA clusters) and its bits follow that
// build's summation order (still the same for every row shard of a chunk).
int mhc_pre_noalloc(const uint16_t *R, const float *fn, const float *scale, const float *base,
                    const uint16_t *norm_w, int64_t rows, int64_t logical_rows,
                    const mhc_params *p, uint16_t *x_norm, float *post, float *comb,
                    float *pre_out, float *mix_out, void *stream) {
  return pre_impl(R, fn, nullptr, scale, base, norm_w, rows, logical_rows, p, nullptr, 0, x_norm,
                  post, comb, pre_out, mix_out, stream, nullptr, nullptr, /*ws_required=*/false);
}

int mhc_post(const uint16_t *R, const uint16_t *y, const float *post, const float *comb,
             int64_t rows, int64_t logical_rows, uint16_t *R_out, void *stream) {
  if (int e = check_rows(rows, logical_rows)) return e;
  if (rows == 0) return MHC_OK;
  if (!R || !y || !post || !comb || !R_out) return MHC_ERR_NULL;
  const void *al[] = {R, y, post, comb, R_out};
  for (const void *q : al)
    if (!aligned16(q)) return MHC_ERR_ALIGN;
  const size_t nr = (size_t)rows;
  const Span out = span(R_out, nr * MHC_K * 2);
  const Span ins[] = {span(R, nr * MHC_K * 2), span(y, nr * MHC_HIDDEN * 2),
                      span(post, nr * MHC_HC * 4), span(comb, nr * MHC_HC * MHC_HC * 4)};
  for (const Span &b : ins)
    if (overlap(out, b)) return MHC_ERR_OVERLAP;
  if (int e = check_device()) return e;
  cudaError_t ce = mhc::launch_post(R, y, post, comb, rows, logical_rows, R_out,
                                    static_cast<cudaStream_t>(stream));
  return ce == cudaSuccess ? MHC_OK : cuda_fail(ce);
}

int mhc_combine_norm(const uint16_t *R, const float *pre, const uint16_t *norm_w,
                     float norm_eps, int64_t rows, int64_t logical_rows, uint16_t *x_norm,
                     void *stream) {
  if (int e = check_rows(rows, logical_rows)) return e;
  if (!finite_nonneg(norm_eps)) return MHC_ERR_PARAM;
  if (rows == 0) return MHC_OK;
  if (!R || !pre || !norm_w || !x_norm) return MHC_ERR_NULL;
  const void *al[] = {R, pre, norm_w, x_norm};
  for (const void *q : al)
    if (!aligned16(q)) return MHC_ERR_ALIGN;
  const size_t nr = (size_t)rows;
  const Span out = span(x_norm, nr * MHC_HIDDEN * 2);
  const Span ins[] = {span(R, nr * MHC_K * 2), span(pre, nr * MHC_HC * 4),
                      span(norm_w, MHC_HIDDEN * 2)};
  for (const Span &b : ins)
    if (overlap(out, b)) return MHC_ERR_OVERLAP;
  if (int e = check_device()) return e;
  cudaError_t ce = mhc::launch_combine_norm(R, pre, norm_w, norm_eps, rows, logical_rows,
                                            x_norm, static_cast<cudaStream_t>(stream));
  return ce == cudaSuccess ? MHC_OK : cuda_fail(ce);
}

namespace {
// mhc_fused_post_pre and its prepared form: fnp_ready is NULL (the call
// writes fn's image into its workspace) or the handle's image (fn is then the
// handle's fp32 copy and the workspace needs no room for an image)
int fused_impl(const uint16_t *R, const uint16_t *y, const float *post, const float *comb,
               const float *fn, const uint8_t *fnp_ready, const float *scale, const float *base,
               const uint16_t *norm_w, int64_t rows, int64_t logical_rows,
               const mhc_params *p_in, void *workspace, size_t workspace_bytes,
               uint16_t *R_out, uint16_t *x_norm, float *post_out, float *comb_out,
               float *pre_out, float *mix_out, void *stream,
               uint8_t *mx_q = nullptr, uint8_t *mx_s = nullptr) {
  mhc_params p;
  if (p_in) p = *p_in; else mhc_default_params(&p);
  if (int e = check_rows(rows, logical_rows)) return e;
  if (!finite_nonneg(p.rms_eps) || !finite_nonneg(p.hc_pre_eps) ||
      !finite_nonneg(p.hc_sinkhorn_eps) || !finite_nonneg(p.norm_eps) ||
      !std::isfinite(p.post_mult) || p.sinkhorn_iters < 1 || p.sinkhorn_iters > 100000)
    return MHC_ERR_PARAM;
  if (rows == 0) return MHC_OK;
  if (!R || !y || !post || !comb || !fn || !scale || !base || !norm_w || !R_out || !x_norm ||
      !post_out || !comb_out)
    return MHC_ERR_NULL;
  const void *al[] = {R, y, post, comb, fn, scale, base, norm_w, R_out, x_norm, post_out, comb_out};
  for (const void *q : al)
    if (!aligned16(q)) return MHC_ERR_ALIGN;
  if ((pre_out && !aligned16(pre_out)) || (mix_out && !aligned16(mix_out))) return MHC_ERR_ALIGN;
  if ((mx_q == nullptr) != (mx_s == nullptr)) return MHC_ERR_NULL;
  if (mx_q && (!aligned16(mx_q) || !aligned16(mx_s))) return MHC_ERR_ALIGN;
  const size_t need = fnp_ready ? mhc_pre_workspace_bytes(rows)
                                : mhc_fused_post_pre_workspace_bytes(rows);
  if (!workspace || workspace_bytes < need || (reinterpret_cast<uintptr_t>(workspace) & 255u))
    return MHC_ERR_WORKSPACE;
  const size_t nr = (size_t)rows;
  const Span ins[] = {span(R, nr * MHC_K * 2), span(y, nr * MHC_HIDDEN * 2),
                      span(post, nr * MHC_HC * 4), span(comb, nr * MHC_HC * MHC_HC * 4),
                      span(fn, (size_t)MHC_MIX * MHC_K * 4), span(scale, 12),
                      span(base, MHC_MIX * 4), span(norm_w, MHC_HIDDEN * 2)};
  Span outs[9];
  int n_out = 0;
  outs[n_out++] = span(R_out, nr * MHC_K * 2);
  outs[n_out++] = span(x_norm, nr * MHC_HIDDEN * 2);
  if (mx_q) {
    outs[n_out++] = span(mx_q, nr * MHC_HIDDEN);
    outs[n_out++] = span(mx_s, nr * (MHC_HIDDEN / 32));
  }
  outs[n_out++] = span(post_out, nr * MHC_HC * 4);
  outs[n_out++] = span(comb_out, nr * MHC_HC * MHC_HC * 4);
  outs[n_out++] = span(workspace, need);
  if (pre_out) outs[n_out++] = span(pre_out, nr * MHC_HC * 4);
  if (mix_out) outs[n_out++] = span(mix_out, nr * MHC_MIX * 4);
  for (int a = 0; a < n_out; ++a) {
    for (const Span &b : ins)
      if (overlap(outs[a], b)) return MHC_ERR_OVERLAP;
    for (int b = a + 1; b < n_out; ++b)
      if (overlap(outs[a], outs[b])) return MHC_ERR_OVERLAP;
  }
  if (int e = check_device()) return e;
  const cudaStream_t s = static_cast<cudaStream_t>(stream);
  cudaError_t ce;
  if (logical_rows <= mhc::kDecodeMaxRows) {
    // decode-size chunk: one launch, hc_post on the loaded columns and the
    // decode pre on R'
    ce = mhc::launch_post_pre_decode(R, y, post, comb, fn, scale, base, norm_w, rows,
                                     logical_rows, p, R_out, x_norm, post_out, comb_out, pre_out,
                                     mix_out, s, /*fn_stable=*/fnp_ready != nullptr);
    // the decode kernel writes bf16 x_norm only; its MXFP8 follows in a
    // second, streaming launch
    if (ce == cudaSuccess && mx_q)
      ce = mhc::launch_mx_quantize(x_norm, rows, MHC_HIDDEN, logical_rows, mx_q, mx_s, s);
  } else {
    float *pre_ws = static_cast<float *>(workspace);
    float *logit_ws = reinterpret_cast<float *>(static_cast<char *>(workspace) + gate_bytes(rows));
    const uint8_t *fnp =
        fnp_ready ? fnp_ready : static_cast<uint8_t *>(workspace) + mhc_pre_workspace_bytes(rows);
    ce = mhc::launch_post_pre_fused(R, y, post, comb, fnp_ready ? nullptr : fn, scale, base, rows,
                                    logical_rows, p, pre_ws, logit_ws, fnp, R_out, post_out,
                                    pre_out, mix_out, s);
    if (ce == cudaSuccess)
      ce = mhc::launch_combine_norm_sinkhorn(R_out, pre_ws, norm_w, p.norm_eps, logit_ws, comb_out,
                                             p.hc_sinkhorn_eps, p.sinkhorn_iters, rows,
                                             logical_rows, x_norm, s, mx_q, mx_s);
  }
  return ce == cudaSuccess ? MHC_OK : cuda_fail(ce);
}
}  // namespace

int mhc_fused_post_pre(const uint16_t *R, const uint16_t *y, const float *post,
                       const float *comb, const float *fn, const float *scale, const float *base,
                       const uint16_t *norm_w, int64_t rows, int64_t logical_rows,
                       const mhc_params *p, void *workspace, size_t workspace_bytes,
                       uint16_t *R_out, uint16_t *x_norm, float *post_out, float *comb_out,
                       float *pre_out, float *mix_out, void *stream) {
  return fused_impl(R, y, post, comb, fn, nullptr, scale, base, norm_w, rows, logical_rows, p,
                    workspace, workspace_bytes, R_out, x_norm, post_out, comb_out, pre_out,
                    mix_out, stream);
}

int mhc_fused_post_pre_prepared(const uint16_t *R, const uint16_t *y, const float *post,
                                const float *comb, const mhc_weights *w, const float *scale,
                                const float *base, const uint16_t *norm_w, int64_t rows,
                                int64_t logical_rows, const mhc_params *p, void *workspace,
                                size_t workspace_bytes, uint16_t *R_out, uint16_t *x_norm,
                                float *post_out, float *comb_out, float *pre_out, float *mix_out,
                                void *stream) {
  if (!w) return MHC_ERR_NULL;
  int dev = -1;
  if (cudaGetDevice(&dev) == cudaSuccess && dev != w->device) return MHC_ERR_DEVICE;
  return fused_impl(R, y, post, comb, w->fn32, w->img64, scale, base, norm_w, rows, logical_rows,
                    p, workspace, workspace_bytes, R_out, x_norm, post_out, comb_out, pre_out,
                    mix_out, stream);
}

int mhc_fused_post_pre_mxfp8(const uint16_t *R, const uint16_t *y, const float *post,
                             const float *comb, const mhc_weights *w, const float *scale,
                             const float *base, const uint16_t *norm_w, int64_t rows,
                             int64_t logical_rows, const mhc_params *p, void *workspace,
                             size_t workspace_bytes, uint16_t *R_out, uint16_t *x_norm,
                             uint8_t *x_q, uint8_t *x_s, float *post_out, float *comb_out,
                             void *stream) {
  if (!w) return MHC_ERR_NULL;
  if (rows > 0 && (!x_q || !x_s)) return MHC_ERR_NULL;
  int dev = -1;
  if (cudaGetDevice(&dev) == cudaSuccess && dev != w->device) return MHC_ERR_DEVICE;
  return fused_impl(R, y, post, comb, w->fn32, w->img64, scale, base, norm_w, rows, logical_rows,
                    p, workspace, workspace_bytes, R_out, x_norm, post_out, comb_out, nullptr,
                    nullptr, stream, x_q, x_s);
}

int mhc_hc_head(const uint16_t *R, const float *fn, const float *scale, const float *base,
                int64_t rows, int64_t logical_rows, float norm_eps, float hc_eps,
                void *workspace, size_t workspace_bytes, uint16_t *y, float *pre_out,
                float *mix_out, void *stream) {
  if (int e = check_rows(rows, logical_rows)) return e;
  if (!finite_nonneg(norm_eps) || !finite_nonneg(hc_eps)) return MHC_ERR_PARAM;
  if (rows == 0) return MHC_OK;
  if (!R || !fn || !scale || !base || !y) return MHC_ERR_NULL;
  const void *al[] = {R, fn, scale, base, y};
  for (const void *q : al)
    if (!aligned16(q)) return MHC_ERR_ALIGN;
  if ((pre_out && !aligned16(pre_out)) || (mix_out && !aligned16(mix_out))) return MHC_ERR_ALIGN;
  const size_t need = mhc_pre_workspace_bytes(rows);
  if (!workspace || workspace_bytes < need || (reinterpret_cast<uintptr_t>(workspace) & 255u))
    return MHC_ERR_WORKSPACE;
  const size_t nr = (size_t)rows;
  const Span ins[] = {span(R, nr * MHC_K * 2), span(fn, (size_t)MHC_HC * MHC_K * 4),
                      span(scale, 4), span(base, MHC_HC * 4)};
  Span outs[4];
  int n_out = 0;
  outs[n_out++] = span(y, nr * MHC_HIDDEN * 2);
  outs[n_out++] = span(workspace, need);
  if (pre_out) outs[n_out++] = span(pre_out, nr * MHC_HC * 4);
  if (mix_out) outs[n_out++] = span(mix_out, nr * MHC_HC * 4);
  for (int a = 0; a < n_out; ++a) {
    for (const Span &b : ins)
      if (overlap(outs[a], b)) return MHC_ERR_OVERLAP;
    for (int b = a + 1; b < n_out; ++b)
      if (overlap(outs[a], outs[b])) return MHC_ERR_OVERLAP;
  }
  if (int e = check_device()) return e;
  const cudaStream_t s = static_cast<cudaStream_t>(stream);
  cudaError_t ce;
  if (logical_rows <= mhc::kHeadOnePassMaxRows) {
    // small chunk: one pass over R on the CUDA cores (no workspace used)
    ce = mhc::launch_head_onepass(R, fn, scale, base, rows, logical_rows, norm_eps, hc_eps, y,
                                  pre_out, mix_out, s);
  } else {
    // one launch: tensor-core stats, the tile kept in shared memory for the
    // combine (no workspace used)
    ce = mhc::launch_head_tile(R, fn, scale, base, rows, logical_rows, norm_eps, hc_eps, y,
                               pre_out, mix_out, s);
  }
  return ce == cudaSuccess ? MHC_OK : cuda_fail(ce);
}

}  // extern "C"
