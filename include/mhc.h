/*
 * mhc.h -- C ABI of libmhc: the row-local manifold-constrained hyper-connection
 * (mHC) work around one sublayer of a DeepSeek-V4 decoder layer, on GB300
 * (sm_103a).
 *
 * The residual R of a chunk of M tokens carries HC = 4 streams of width
 * H = 5120 (R[M, 4, 5120], bf16).  Around every sublayer the model runs
 *   pre : stats -> split/Sinkhorn -> combine + RMSNorm  (feeds the sublayer)
 *   post: new residual from the sublayer output          (after the sublayer)
 * as defined in deepseek_v4.py (sglang), DeepseekV4DecoderLayer.hc_pre and
 * DeepseekV4DecoderLayer.hc_post.  Beside mhc_pre and mhc_post: the two fused
 * across a sublayer boundary (mhc_fused_post_pre), the model's final stream
 * collapse (mhc_hc_head), prepared weights (mhc_prepare_weights and the
 * *_prepared calls) and MXFP8 output of the normalised input (mhc_pre_mxfp8,
 * mhc_quantize_mxfp8, mhc_swizzle_scales_128x4).
 *
 * Conventions for every entry point below
 *  - All tensor arguments are DEVICE pointers, owned by the caller, row-major
 *    and densely packed in the layout stated; bf16 tensors are passed as
 *    uint16_t bit patterns.  Every tensor pointer must be 16-byte aligned.
 *  - Calls are asynchronous: they enqueue kernels on `stream` (a
 *    cudaStream_t; NULL means the legacy default stream) and never
 *    synchronise.  Device-side faults surface at the caller's next
 *    synchronisation, as with any CUDA launch.
 *  - For chunks of at most 2048 rows (logical_rows) the kernels are launched
 *    with programmatic stream serialization: a kernel's blocks may be
 *    scheduled before the previous work on the stream has finished, but each
 *    waits for it to complete (griddepcontrol.wait) before touching memory,
 *    so stream order holds for every caller.  It also holds under stream
 *    capture.
 *  - `rows` is the number of rows this call processes (a row-range shard
 *    passes pointers already offset to its first row).  `logical_rows` is
 *    the row count of the whole chunk the rows belong to; launch heuristics
 *    may read only `logical_rows`, never `rows`, so any row range
 *    [lo, hi) of a chunk gives exactly the bits the whole-chunk call gives
 *    on those rows (prefill_sp.py, sp_logical_rows: kernel gates key on the
 *    full chunk row count).  logical_rows >= rows is required.
 *  - rows == 0 returns MHC_OK without launching anything.
 *  - Arguments are validated on the host before any launch; on an error the
 *    call returns a negative code, launches nothing and writes nothing.
 *  - Output buffers must not overlap any input buffer.
 *  - No call allocates device memory except mhc_prepare_weights (its
 *    handle's 5.9 MB, freed by mhc_release_weights).  Scratch space, where an
 *    entry point needs it, is passed in by the caller (`workspace`), except
 *    for mhc_pre_noalloc, whose kernels need none.
 */
#ifndef MHC_H
#define MHC_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define MHC_HC 4                       /* hc_mult: residual streams */
#define MHC_HIDDEN 5120                /* hidden size H */
#define MHC_K (MHC_HC * MHC_HIDDEN)    /* flattened row width 20480 */
#define MHC_MIX 24                     /* (2 + hc_mult) * hc_mult mixes */

/* return codes */
#define MHC_OK 0
#define MHC_ERR_NULL (-1)        /* a required pointer is NULL */
#define MHC_ERR_SHAPE (-2)       /* rows < 0, logical_rows < rows, rows too large, or a bad column / group count */
#define MHC_ERR_ALIGN (-3)       /* a tensor pointer is not 16-byte aligned */
#define MHC_ERR_PARAM (-4)       /* eps < 0 or not finite, iters < 1, ... */
#define MHC_ERR_OVERLAP (-5)     /* an output buffer overlaps an input buffer */
#define MHC_ERR_WORKSPACE (-6)   /* workspace NULL or smaller than required */
#define MHC_ERR_CUDA (-7)        /* a CUDA call failed (see mhc_last_cuda_error) */
#define MHC_ERR_DEVICE (-8)      /* current device is not an sm_103 GPU */
#define MHC_ERR_SCRATCH_LIMIT (-9) /* reserved: no entry point of this build returns it */
#define MHC_ERR_ALLOC (-10)      /* a device allocation failed (mhc_prepare_weights) */

/* Scalars of the split/Sinkhorn and the two RMS normalisations.
 * deepseek_v4.py, DeepseekV4DecoderLayer.hc_pre passes rms_eps =
 * rms_norm_eps, hc_pre_eps = hc_sinkhorn_eps = hc_eps, post_mult =
 * _MHC_POST_MULT_VALUE (2.0) and sinkhorn_repeat = hc_sinkhorn_iters;
 * norm_eps is the RMSNorm's variance epsilon. */
typedef struct mhc_params {
    float rms_eps;          /* added to mean(x^2) of the flattened row (stats) */
    float hc_pre_eps;       /* pre = sigmoid(logit) + hc_pre_eps */
    float hc_sinkhorn_eps;  /* added to every Sinkhorn row and column sum */
    float norm_eps;         /* RMSNorm: added to mean(y^2) */
    float post_mult;        /* post = post_mult * sigmoid(logit) */
    int32_t sinkhorn_iters; /* full row+column normalisation rounds, >= 1 */
} mhc_params;

/* Fill *p with rms_eps = hc_pre_eps = hc_sinkhorn_eps = norm_eps = 1e-6,
 * post_mult = 2, sinkhorn_iters = 20 (the values test_prefill_sp_gpu.py's
 * Layer stand-in uses). */
void mhc_default_params(mhc_params *p);

/* Static description of a return code; never NULL. */
const char *mhc_strerror(int code);

/* Text of the last CUDA error seen by this thread inside libmhc ("" if none). */
const char *mhc_last_cuda_error(void);

/* Bytes of device scratch mhc_pre, mhc_hc_head and mhc_fused_post_pre take
 * for a call on `rows` rows (0 for rows <= 0): the larger of
 *   - fn's operand image, 1,966,080 bytes: mhc_pre writes it there for a
 *     chunk of 2048 rows or more (logical_rows), whose one-pass launch
 *     streams it (see mhc_pre);
 *   - the pre gates [rows, 4] fp32 and the comb logits [rows, 16] fp32 that
 *     mhc_fused_post_pre's tensor-core launch hands its combine launch, each
 *     rounded up to 256 bytes.
 * mhc_hc_head and the decode-size paths use none of it. */
size_t mhc_pre_workspace_bytes(int64_t rows);

/* Read libmhc's device status word on the current device into *status: 0,
 * or nonzero once a cluster kernel (of mhc_pre, mhc_hc_head or
 * mhc_fused_post_pre, at any size) gave up a bounded wait (it then returned
 * early, or finished on what had landed: its outputs are incomplete).
 * reset != 0 clears it.  Synchronous: waits for
 * the device's pending work.  Returns MHC_OK or MHC_ERR_NULL/MHC_ERR_CUDA. */
int mhc_kernel_status(uint32_t *status, int reset);

/* Where the waits of mhc_pre's one-pass kernel ended, for diagnosis: bit s
 * (s < 16) of its error word means a bounded wait at site s expired, bit
 * 16 + s that a wait at site s gave up because its CTA had already aborted.
 * where64[s] (expired) and where64[32 + s] (gave up) hold (tile << 8) | CTA
 * rank in its cluster of the last such event.  where64 has 64 entries.
 * Synchronous. */
int mhc_kernel_status_detail(uint32_t *where64);

/*
 * mhc_pre -- stats, split/Sinkhorn, combine + RMSNorm for `rows` rows.
 *
 * deepseek_v4.py, DeepseekV4DecoderLayer.hc_pre: with x = R[m] flattened
 * stream-major (k = i*5120 + h) in fp32,
 *   rsqrt     = 1 / sqrt(mean_k x_k^2 + rms_eps)
 *   mix[c]    = rsqrt * sum_k x_k * fn[c, k]                     (c < 24)
 *   logit[c]  = mix[c] * scale[g(c)] + base[c],  g = 0 | 1 | 2 for
 *               c in [0,4) | [4,8) | [8,24)
 *   pre[i]    = sigmoid(logit[i]) + hc_pre_eps
 *   post[i]   = post_mult * sigmoid(logit[4+i])
 *   comb      = exp(logit[8 + 4j + i]) as comb[j][i], then sinkhorn_iters
 *               rounds of: divide row j by (sum_i comb[j][i] + eps), then
 *               column i by (sum_j comb[j][i] + eps)  (hc_split_sinkhorn)
 *   y[h]      = sum_i pre[i] * R[m, i, h]                        (fp32)
 *   x_norm[h] = bf16( y[h] / sqrt(mean_h y^2 + norm_eps) * w[h] )
 * (RMSNorm fused without rounding y first, as the fused combine+norm gate of
 * prefill_sp.py, _combine_norm_fused, requires.)
 *
 * Chunks of more than 48 rows (logical_rows > 48) take one launch that reads
 * R from HBM once (pre_onepass.cu): a cluster of CTAs splits each 32-row
 * tile by hidden columns, streams R with TMA, runs the 24 projections and each
 * row's 4x4 stream Gram matrix on the tensor cores (fn split into bf16 hi +
 * lo), exchanges the partial sums between the CTAs of the cluster, finalises
 * gates, Sinkhorn and 1/rms(y) = 1/sqrt(p^T G p / 5120 + norm_eps), and
 * combines the tile's columns again from L2.  Below 2048 logical rows the
 * clusters have 16 CTAs, which convert fn's operand tiles into shared memory
 * (mhc_pre) or stream them from the prepared image (mhc_pre_prepared); from
 * 2048 rows on they have 8 CTAs (120 SMs busy instead of 112) that stream
 * fn's tiles from an image beside R, and mhc_pre first writes that image (a
 * conversion launch) into the workspace.  Every row's arithmetic is the same
 * whichever source fn comes from.  Decode-size chunks
 * (logical_rows <= 48) take one latency-shaped launch (pre_decode.cu):
 * 16-CTA clusters of CUDA-core work, a group of up to 8 rows per cluster;
 * they do not touch the workspace.
 *
 * Arguments
 *   R        [rows, 4, 5120] bf16      residual rows
 *   fn       [24, 20480] fp32          hc_fn mixing projection
 *   scale    [3] fp32                  hc_scale (pre, post, comb)
 *   base     [24] fp32                 hc_base
 *   norm_w   [5120] bf16               RMSNorm weight
 *   p        host pointer; NULL means mhc_default_params
 *   workspace, workspace_bytes  device scratch of at least
 *            mhc_pre_workspace_bytes(rows) bytes, 256-byte aligned; its
 *            contents on entry do not matter; the call owns it until the
 *            stream reaches the end of the call.  Written (fn's image) only
 *            by chunks of 2048 rows or more.
 * Outputs (fp32 unless stated)
 *   x_norm   [rows, 5120] bf16         normalised combine (sublayer input)
 *   post     [rows, 4]                 post gate
 *   comb     [rows, 4, 4]              Sinkhorn mix, comb[m][j][i]
 *   pre_out  [rows, 4] or NULL         pre gate
 *   mix_out  [rows, 24] or NULL        mix (after rsqrt scaling)
 */
int mhc_pre(const uint16_t *R, const float *fn, const float *scale, const float *base,
            const uint16_t *norm_w, int64_t rows, int64_t logical_rows, const mhc_params *p,
            void *workspace, size_t workspace_bytes, uint16_t *x_norm, float *post,
            float *comb, float *pre_out, float *mix_out, void *stream);

/*
 * mhc_pre_noalloc -- mhc_pre for callers that cannot provide device scratch.
 *
 * The pages have no counterpart to this entry point; it exists for callers
 * that cannot allocate device memory on this library's behalf: a framework
 * whose caching allocator owns the device memory, a plugin/operator enqueue
 * that must not allocate, a latency-critical serving loop that cannot afford
 * cudaMalloc/cudaFree (they may synchronise the device), or a C/FFI caller
 * with no device allocator.
 *
 * Same arguments, outputs and validation as mhc_pre, minus the workspace.
 * Below 2048 logical rows it runs exactly mhc_pre's launches (the
 * decode-size launch up to 48 logical rows, the one-pass launch above) and
 * gives mhc_pre's bits.  From 2048 rows on, with no scratch for fn's image,
 * it runs the one-pass launch that keeps fn's tiles resident (16-CTA
 * clusters): the same outputs to within fp32 summation order (the oracle's
 * tolerances), and every row range of a chunk still gives the whole-chunk
 * bits.  It allocates nothing (no cudaMalloc, no cudaFree,
 * no allocating library call) and holds no state between calls, so calls on
 * any streams or host threads may overlap.  mhc_pre_noalloc_max_rows()
 * returns the library-wide row limit (2^24).
 */
int mhc_pre_noalloc(const uint16_t *R, const float *fn, const float *scale, const float *base,
                    const uint16_t *norm_w, int64_t rows, int64_t logical_rows,
                    const mhc_params *p, uint16_t *x_norm, float *post, float *comb,
                    float *pre_out, float *mix_out, void *stream);

/* Largest `rows` mhc_pre_noalloc accepts (2^24, as every entry point). */
int64_t mhc_pre_noalloc_max_rows(void);

/*
 * mhc_post -- the new residual after a sublayer.
 *
 * deepseek_v4.py, DeepseekV4DecoderLayer.hc_post (hc_post_torch_impl):
 *   R_out[m, i, h] = bf16( post[m, i] * y[m, h] + sum_j comb[m, j, i] * R[m, j, h] )
 * computed in fp32 and rounded once.
 *   R      [rows, 4, 5120] bf16   residual that entered the sublayer
 *   y      [rows, 5120] bf16      sublayer output
 *   post   [rows, 4] fp32, comb [rows, 4, 4] fp32 (as mhc_pre wrote them)
 *   R_out  [rows, 4, 5120] bf16   output; must not overlap any input
 */
int mhc_post(const uint16_t *R, const uint16_t *y, const float *post, const float *comb,
             int64_t rows, int64_t logical_rows, uint16_t *R_out, void *stream);

/*
 * mhc_combine_norm -- the combine + RMSNorm step alone, with a given pre.
 *
 * deepseek_v4.py, DeepseekV4DecoderLayer.hc_pre (combine after
 * hc_split_sinkhorn) fused with RMSNorm as in prefill_sp.py,
 * hc_combine_norm_rows:
 *   x_norm[m, h] = bf16( y[h] / sqrt(mean_h y^2 + norm_eps) * w[h] ),
 *   y[h] = sum_i pre[m, i] * R[m, i, h].
 *   R [rows, 4, 5120] bf16, pre [rows, 4] fp32, norm_w [5120] bf16,
 *   x_norm [rows, 5120] bf16.  norm_eps >= 0 and finite.
 */
int mhc_combine_norm(const uint16_t *R, const float *pre, const uint16_t *norm_w,
                     float norm_eps, int64_t rows, int64_t logical_rows, uint16_t *x_norm,
                     void *stream);

/*
 * Prepared weights -- a layer's fn converted once, at load time, into what the
 * kernels read, so that mhc_pre does not convert it at every call.
 *
 * deepseek_v4.py: DeepseekV4DecoderLayer.refresh_mhc_norm_weight_cache casts
 * the norm weights once so the fused path does not cast per forward, and
 * DeepseekV4ForCausalLM._prewarm_mhc_pre_kernels sets mhc_pre up at load
 * time; the handle does the same for fn.
 *
 * mhc_prepare_weights(fn, &w, stream)
 *   fn [24, 20480] fp32, device, 16-byte aligned (hc_fn of one sublayer).
 *   Allocates device memory on the current device (about 5.9 MB, the only
 *   allocation libmhc makes) and enqueues on `stream`: a copy of fn, and
 *   fn's bf16 hi/lo operand images for the one-pass pre kernel and for the
 *   fused post -> pre kernel (the same bits those kernels would form
 *   themselves).  The handle may be
 *   used by calls enqueued after it on `stream`, or on any stream once the
 *   caller has ordered them after it; fn itself may be freed or changed
 *   afterwards.  Returns MHC_OK, MHC_ERR_NULL, MHC_ERR_ALIGN, MHC_ERR_DEVICE,
 *   MHC_ERR_ALLOC (then *out = NULL) or MHC_ERR_CUDA.
 * mhc_release_weights(w)
 *   Frees the handle (NULL is a no-op).  No work using it may still be
 *   pending.
 * mhc_pre_prepared(R, w, scale, base, norm_w, ...)
 *   mhc_pre with fn taken from the handle: the same arguments, checks and
 *   outputs, bit-identical to mhc_pre on the fn the handle was made from.
 *   MHC_ERR_DEVICE if the current device is not the handle's.
 * mhc_fused_post_pre_prepared(R, y, post, comb, w, scale, base, norm_w, ...)
 *   mhc_fused_post_pre likewise (w is the next sublayer's weights); its
 *   workspace needs only mhc_pre_workspace_bytes(rows) bytes, since the call
 *   no longer converts fn.
 */
typedef struct mhc_weights mhc_weights;
int mhc_prepare_weights(const float *fn, mhc_weights **out, void *stream);
int mhc_release_weights(mhc_weights *w);
int mhc_pre_prepared(const uint16_t *R, const mhc_weights *w, const float *scale,
                     const float *base, const uint16_t *norm_w, int64_t rows,
                     int64_t logical_rows, const mhc_params *p, void *workspace,
                     size_t workspace_bytes, uint16_t *x_norm, float *post, float *comb,
                     float *pre_out, float *mix_out, void *stream);
int mhc_fused_post_pre_prepared(const uint16_t *R, const uint16_t *y, const float *post,
                                const float *comb, const mhc_weights *w, const float *scale,
                                const float *base, const uint16_t *norm_w, int64_t rows,
                                int64_t logical_rows, const mhc_params *p, void *workspace,
                                size_t workspace_bytes, uint16_t *R_out, uint16_t *x_norm,
                                float *post_out, float *comb_out, float *pre_out, float *mix_out,
                                void *stream);

/*
 * mhc_fused_post_pre -- hc_post of one sublayer and hc_pre of the next on its
 * result, in one call (the pages' mhc_fused_post_pre between sublayers).
 *
 * deepseek_v4.py, DeepseekV4DecoderLayer forward (the use_fused_mhc_post_pre
 * path): R_out = hc_post(R, y, post, comb) exactly as mhc_post computes it
 * (same bits), then everything mhc_pre computes, on R_out, with the next
 * sublayer's fn, scale, base and norm weight.
 *
 * Chunks of more than 48 rows: a short launch converts fn into the fused
 * kernel's operand image, then one launch computes R_out, writes it once and
 * feeds it straight to the tensor-core stats (R_out is never read back for
 * them), then the pre pass's streaming combine + RMSNorm (with the Sinkhorn)
 * reads R_out.  Decode-size chunks (<= 48 rows): one launch of the decode
 * kernel that forms R_out on the columns it loads and runs mhc_pre on it
 * (R_out and every output bit-identical to mhc_post then mhc_pre).
 *
 * Arguments
 *   R, y, post, comb        as for mhc_post (post [rows, 4] and comb
 *                           [rows, 4, 4] of the sublayer just run)
 *   fn, scale, base, norm_w as for mhc_pre (of the next sublayer)
 *   p        as for mhc_pre
 *   workspace, workspace_bytes  device scratch of at least
 *            mhc_fused_post_pre_workspace_bytes(rows) bytes, 256-byte aligned
 *            (what the pre launches hand each other, plus fn converted by the
 *            call into the fused kernel's operand image, 1.97 MB)
 * Outputs
 *   R_out    [rows, 4, 5120] bf16   the new residual
 *   x_norm   [rows, 5120] bf16      the next sublayer's input
 *   post_out [rows, 4], comb_out [rows, 4, 4] fp32   the next sublayer's gates
 *   pre_out  [rows, 4] or NULL, mix_out [rows, 24] or NULL
 * No output may overlap an input or another output.  Errors as for mhc_pre.
 */
size_t mhc_fused_post_pre_workspace_bytes(int64_t rows);
int mhc_fused_post_pre(const uint16_t *R, const uint16_t *y, const float *post,
                       const float *comb, const float *fn, const float *scale, const float *base,
                       const uint16_t *norm_w, int64_t rows, int64_t logical_rows,
                       const mhc_params *p, void *workspace, size_t workspace_bytes,
                       uint16_t *R_out, uint16_t *x_norm, float *post_out, float *comb_out,
                       float *pre_out, float *mix_out, void *stream);

/*
 * mhc_hc_head -- the model's final collapse of the 4 residual streams into one
 * hidden state (run once per forward, after the last decoder layer and before
 * the final norm).
 *
 * deepseek_v4.py, make_hc_head_params and hc_head_torch: with x = R[m]
 * flattened stream-major in fp32,
 *   rsqrt  = 1 / sqrt(mean_k x_k^2 + norm_eps)
 *   mix[i] = rsqrt * sum_k x_k * fn[i, k]                      (i < 4)
 *   pre[i] = sigmoid(mix[i] * scale[0] + base[i]) + hc_eps
 *   y[m,h] = bf16( sum_i pre[i] * R[m, i, h] )     (fp32 sum, one rounding)
 *
 * One launch that reads R once and combines every row from shared memory.
 * Chunks of more than 256 rows (logical_rows): 8-CTA clusters over 16-row
 * tiles (head_tile.cu), the 4 dots on the tensor cores against fn split
 * into bf16 hi + lo, the tile kept in an 11-stage shared-memory ring until
 * its gates come back.  Chunks of up to 256 rows: 4-CTA clusters that form
 * the 4 dots in fp32 on the CUDA cores (head_onepass.cu).  The two paths
 * form the dots differently and agree to the gate tolerance; every row
 * range of a chunk gives the whole-chunk bits.  Neither uses the workspace,
 * which is validated as for mhc_pre (mhc_pre_workspace_bytes(rows)).
 *
 * Arguments
 *   R        [rows, 4, 5120] bf16      residual after the last layer
 *   fn       [4, 20480] fp32           hc_head_fn
 *   scale    [1] fp32                  hc_head_scale
 *   base     [4] fp32                  hc_head_base
 *   norm_eps, hc_eps                   >= 0 and finite (the model's norm_eps
 *                                      and hc_eps)
 *   workspace, workspace_bytes  as for mhc_pre: at least
 *            mhc_pre_workspace_bytes(rows) bytes, 256-byte aligned.
 * Outputs
 *   y        [rows, 5120] bf16         collapsed hidden state
 *   pre_out  [rows, 4] fp32 or NULL    the gates
 *   mix_out  [rows, 4] fp32 or NULL    the mixes (after rsqrt scaling)
 * Errors as for mhc_pre.
 */
int mhc_hc_head(const uint16_t *R, const float *fn, const float *scale, const float *base,
                int64_t rows, int64_t logical_rows, float norm_eps, float hc_eps,
                void *workspace, size_t workspace_bytes, uint16_t *y, float *pre_out,
                float *mix_out, void *stream);

/*
 * MXFP8 output of x_norm -- the attention input as fp8 codes with one
 * power-of-two scale per 32 values.
 *
 * prefill_sp.py, _mxfp8_quantize and mxfp8_gather: each rank quantizes its
 * bf16 rows per row and per 32 columns (linear scale layout), and
 * swizzle_128x4 tiles the chunk's scales for the GEMM that reads them.  The
 * pages call a library quantizer and do not state its rule; libmhc takes the
 * OCP Microscaling Formats (MX) v1.0 conversion to E4M3:
 *   amax = max |x| over the block (x as bf16, i.e. x_norm's stored values)
 *   e    = floor(log2 amax) - 8, at least -127 (e = -127 for amax = 0)
 *   s    = e + 127                     ue8m0 code of the scale 2^e
 *   q_k  = E4M3(x_k / 2^e)             round to nearest-even, saturate to
 *                                      +-448, sign kept (-0 gives 0x80)
 * Values must be finite.
 *
 * mhc_pre_mxfp8(R, w, scale, base, norm_w, rows, logical_rows, p, workspace,
 *               workspace_bytes, x_norm, x_q, x_s, post, comb, stream)
 *   mhc_pre_prepared (same arguments, checks and bits) that also writes
 *   x_q [rows, 5120] uint8 E4M3 codes and x_s [rows, 160] uint8 scales of
 *   x_norm, both device, 16-byte aligned, overlapping nothing else.  Chunks
 *   of more than 48 rows: the one-pass kernel's combine writes them beside
 *   x_norm; decode-size chunks: one more launch after the decode kernel.
 *   MHC_ERR_NULL if x_q or x_s is NULL.
 * mhc_fused_post_pre_mxfp8(R, y, post, comb, w, scale, base, norm_w, rows,
 *               logical_rows, p, workspace, workspace_bytes, R_out, x_norm,
 *               x_q, x_s, post_out, comb_out, stream)
 *   mhc_fused_post_pre_prepared (same arguments, checks and bits, without
 *   pre_out/mix_out) that also writes x_q [rows, 5120] and x_s [rows, 160]
 *   of the next sublayer's x_norm, as mhc_pre_mxfp8 does: above 48 rows the
 *   fused call's combine launch writes them beside x_norm, at decode sizes one more
 *   launch follows the fused decode kernel.  MHC_ERR_NULL if x_q or x_s is
 *   NULL.
 * mhc_quantize_mxfp8(x, rows, cols, logical_rows, q, s, stream)
 *   The same quantization of any bf16 rows: x [rows, cols] bf16 (cols a
 *   multiple of 32, at most 65536), q [rows, cols] uint8, s [rows, cols/32]
 *   uint8 (linear layout), all device, 16-byte aligned, no overlap.
 *   logical_rows as for mhc_pre (launch shape only).  MHC_ERR_SHAPE for a
 *   bad rows/cols; rows = 0 launches nothing.
 * mhc_swizzle_scales_128x4(s, rows, groups, out, stream)
 *   s [rows, groups] uint8 linear scales (groups a multiple of 4, at most
 *   2048) -> out, mhc_swizzle_scales_128x4_bytes(rows, groups) =
 *   ceil(rows/128)*128*groups bytes: rows padded with zero scales to a
 *   multiple of 128; tile (m/128, g/4) is the (m/128 * groups/4 + g/4)-th
 *   run of 512 bytes, inside which (m, g) sits at byte
 *   (m%32)*16 + ((m%128)/32)*4 + g%4.  Device buffers, 16-byte aligned, not
 *   overlapping.  Run it on the whole chunk's scales (a shard's rows do not
 *   in general fill whole 128-row tiles).
 * All enqueue on `stream` and return MHC_OK or an MHC_ERR_* code, as mhc_pre.
 */
int mhc_pre_mxfp8(const uint16_t *R, const mhc_weights *w, const float *scale, const float *base,
                  const uint16_t *norm_w, int64_t rows, int64_t logical_rows,
                  const mhc_params *p, void *workspace, size_t workspace_bytes,
                  uint16_t *x_norm, uint8_t *x_q, uint8_t *x_s, float *post, float *comb,
                  void *stream);
int mhc_fused_post_pre_mxfp8(const uint16_t *R, const uint16_t *y, const float *post,
                             const float *comb, const mhc_weights *w, const float *scale,
                             const float *base, const uint16_t *norm_w, int64_t rows,
                             int64_t logical_rows, const mhc_params *p, void *workspace,
                             size_t workspace_bytes, uint16_t *R_out, uint16_t *x_norm,
                             uint8_t *x_q, uint8_t *x_s, float *post_out, float *comb_out,
                             void *stream);
int mhc_quantize_mxfp8(const uint16_t *x, int64_t rows, int64_t cols, int64_t logical_rows,
                       uint8_t *q, uint8_t *s, void *stream);
size_t mhc_swizzle_scales_128x4_bytes(int64_t rows, int64_t groups);
int mhc_swizzle_scales_128x4(const uint8_t *s, int64_t rows, int64_t groups, uint8_t *out,
                             void *stream);

#ifdef __cplusplus
}
#endif

#endif /* MHC_H */
