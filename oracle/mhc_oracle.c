/*
 * mhc_oracle.c -- plain, slow, single-threaded CPU oracle of the row-local
 * hyper-connection (mHC) work around one sublayer of a DeepSeek-V4 decoder.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product path (the CUDA library
 * and its Python binding) may include, link or call this file.  Only the
 * tests, the smoke check and the benchmark's CPU-baseline leg use it.  It
 * shares no code, header, table or constant generator with the CUDA path.
 *
 * Arithmetic: every input (bf16 bits or fp32) is widened exactly to double;
 * all sums, products, exp, sqrt and divisions are done in double in the
 * plain order written below; each bf16 output is rounded once, directly from
 * double, to nearest-even.
 *
 * Sources (page title, section):
 *   deepseek_v4.py (sglang), DeepseekV4DecoderLayer.hc_pre,
 *     inner hc_pre_torch_impl: x = R.flatten(1).float();
 *     rsqrt(mean(x^2) + rms_norm_eps); mixes = (x @ fn^T) * rsqrt.
 *   deepseek_v4.py, DeepseekV4DecoderLayer.hc_pre, tail:
 *     pre, post, comb = hc_split_sinkhorn(mixes, scale, base, hc_mult,
 *     iters, hc_eps); y = sum_i pre_i * x.view(M,4,H)[:, i, :].
 *   deepseek_v4.py, module constants: _MHC_POST_MULT_VALUE = 2.0;
 *     make_hc_mixing_params: fn [24, 4H], base [24], scale [3].
 *   deepseek_v4.py, hc_head_torch: pre = sigmoid(mixes*scale + base) + hc_eps
 *     (the "sigmoid + eps" pattern the pre gate follows).
 *   deepseek_v4.py, DeepseekV4DecoderLayer.hc_post, inner hc_post_torch_impl:
 *     R'[:, i, :] = post_i * y + sum_j comb[:, j, i] * R[:, j, :].
 *   prefill_sp.py, _combine_norm_fused: the fused combine+RMSNorm kernel is
 *     used only when the norm does not cast x before the weight multiply.
 *   deepseek_v4.py, make_hc_head_params and hc_head_torch: the model's final
 *     collapse of the 4 streams, fn [4, 4H], base [4], scale [1];
 *     rsqrt(mean(x^2) + norm_eps); pre = sigmoid(mixes*scale + base) + hc_eps;
 *     y = sum_i pre_i * x_i, cast once to the residual's dtype.
 *
 * The body of hc_split_sinkhorn is not on the pages.  The reading used here
 * (each choice is one reading of an open step, not a fact of the pages):
 *   - the 24 mixes split in order [0,4) pre, [4,8) post, [8,24) comb, the
 *     comb block row-major as comb[j][i] = mix[8 + 4*j + i];
 *   - logit_c = mix_c * scale[g] + base_c with g = 0, 1, 2 for pre, post,
 *     comb;
 *   - pre_i = sigmoid(logit_i) + hc_pre_eps; post_i = post_mult *
 *     sigmoid(logit_{4+i}) (no eps);
 *   - comb starts as exp(logit) (no max subtraction) and each of the `iters`
 *     iterations first divides every row j by (its sum over i + eps), then
 *     every column i by (its sum over j + eps).
 * The combine+RMSNorm keeps y in full precision (fused reading); an option
 * emulates the unfused path, which rounds y to bf16 before the norm.
 *
 * MXFP8 output of x_norm (prefill_sp.py, _mxfp8_quantize / mxfp8_gather and
 * swizzle_128x4): per row, per 32 columns, fp8 codes plus one ue8m0 scale,
 * scales in a linear [rows, cols/32] layout, and the 128x4 tiled scale layout
 * the pages build from it.  The pages call a library quantizer and do not
 * state its scale or rounding rule; the reading used here is the OCP
 * Microscaling Formats (MX) v1.0 conversion: shared exponent
 * floor(log2(block amax)) - 8 (8 = the largest exponent of E4M3), clamped to
 * the scale format's range, elements x / 2^shared rounded to E4M3 nearest-even
 * and saturated to +-448, the sign kept (so -0 and tiny negatives give 0x80).
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define O_HC 4
#define O_H 5120
#define O_K (O_HC * O_H)
#define O_MIX 24

/* ---- exact bf16 <-> double ------------------------------------------------ */

double oracle_bf16_to_double(uint16_t b)
{
    uint32_t u = (uint32_t)b << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

/* Round a double to the nearest bf16 (ties to even), in one step.  bf16 has
 * an 8-bit significand and float's exponent range; the quantum of a normal
 * value in [2^(e-1), 2^e) is 2^(e-8), and of subnormals 2^-133. */
uint16_t oracle_double_to_bf16(double d)
{
    if (isnan(d))
        return 0x7FC0;
    uint16_t sign = signbit(d) ? 0x8000 : 0;
    double a = fabs(d);
    if (a == 0.0)
        return sign;
    if (isinf(a))
        return sign | 0x7F80;
    int e;
    (void)frexp(a, &e);           /* a = f * 2^e, f in [0.5, 1) */
    int q = e - 8;                /* quantum exponent */
    if (q < -133)
        q = -133;
    double s = ldexp(a, -q);      /* exact: scaling by a power of two */
    double r = nearbyint(s);      /* default rounding mode: nearest, ties even */
    double v = ldexp(r, q);
    if (v > 3.3895313892515355e38) /* largest finite bf16 */
        return sign | 0x7F80;
    float f = (float)v;           /* exact: v has at most 8 significant bits */
    uint32_t u;
    memcpy(&u, &f, sizeof u);
    return sign | (uint16_t)(u >> 16);
}

/* ---- a1: mix stats -------------------------------------------------------- */

/* For each row m of R[rows, 4, 5120] (bf16 bits), with x = R[m] flattened
 * stream-major (k = i*5120 + h):
 *   rsq[m]      = 1 / sqrt( (sum_k x_k^2) / 20480 + rms_eps )
 *   mix[m, c]   = rsq[m] * sum_k x_k * fn[c, k]        (c = 0..23)
 * fn is [24, 20480] fp32. */
void oracle_stats(const uint16_t *R, int64_t rows, const float *fn, double rms_eps,
                  double *mix, double *rsq)
{
    double *x = (double *)malloc(sizeof(double) * O_K);
    for (int64_t m = 0; m < rows; ++m) {
        const uint16_t *row = R + m * (int64_t)O_K;
        double ss = 0.0;
        for (int k = 0; k < O_K; ++k) {
            x[k] = oracle_bf16_to_double(row[k]);
            ss += x[k] * x[k];
        }
        double r = 1.0 / sqrt(ss / (double)O_K + rms_eps);
        if (rsq)
            rsq[m] = r;
        for (int c = 0; c < O_MIX; ++c) {
            const float *f = fn + (int64_t)c * O_K;
            double dot = 0.0;
            for (int k = 0; k < O_K; ++k)
                dot += x[k] * (double)f[k];
            mix[m * O_MIX + c] = dot * r;
        }
    }
    free(x);
}

/* ---- a2 + a3: split, gates, Sinkhorn ------------------------------------- */

static double sigmoid(double z) { return 1.0 / (1.0 + exp(-z)); }

/* mix [rows, 24] -> logits [rows, 24], pre [rows, 4], post [rows, 4],
 * comb [rows, 4, 4] laid out comb[m][j][i]. */
void oracle_split_sinkhorn(const double *mix, int64_t rows, const float *scale,
                           const float *base, double pre_eps, double sink_eps,
                           double post_mult, int iters, double *logits, double *pre,
                           double *post, double *comb)
{
    for (int64_t m = 0; m < rows; ++m) {
        double l[O_MIX];
        for (int c = 0; c < O_MIX; ++c) {
            int g = c < 4 ? 0 : (c < 8 ? 1 : 2);
            l[c] = mix[m * O_MIX + c] * (double)scale[g] + (double)base[c];
            if (logits)
                logits[m * O_MIX + c] = l[c];
        }
        for (int i = 0; i < O_HC; ++i) {
            pre[m * O_HC + i] = sigmoid(l[i]) + pre_eps;
            post[m * O_HC + i] = post_mult * sigmoid(l[4 + i]);
        }
        double C[O_HC][O_HC];
        for (int j = 0; j < O_HC; ++j)
            for (int i = 0; i < O_HC; ++i)
                C[j][i] = exp(l[8 + 4 * j + i]);
        for (int t = 0; t < iters; ++t) {
            for (int j = 0; j < O_HC; ++j) {          /* rows: sum over i */
                double s = 0.0;
                for (int i = 0; i < O_HC; ++i)
                    s += C[j][i];
                for (int i = 0; i < O_HC; ++i)
                    C[j][i] = C[j][i] / (s + sink_eps);
            }
            for (int i = 0; i < O_HC; ++i) {          /* columns: sum over j */
                double s = 0.0;
                for (int j = 0; j < O_HC; ++j)
                    s += C[j][i];
                for (int j = 0; j < O_HC; ++j)
                    C[j][i] = C[j][i] / (s + sink_eps);
            }
        }
        for (int j = 0; j < O_HC; ++j)
            for (int i = 0; i < O_HC; ++i)
                comb[m * 16 + j * 4 + i] = C[j][i];
    }
}

/* ---- a4: combine + RMSNorm ------------------------------------------------ */

/* y[h] = sum_i pre[m, i] * R[m, i, h];
 * x_norm[m, h] = bf16( y[h] / sqrt(mean_h y^2 + norm_eps) * w[h] ).
 * round_y != 0 rounds y to bf16 first (the unfused combine-then-norm path). */
void oracle_combine_norm(const uint16_t *R, int64_t rows, const double *pre,
                         const uint16_t *w, double norm_eps, int round_y, uint16_t *x_norm)
{
    double *y = (double *)malloc(sizeof(double) * O_H);
    for (int64_t m = 0; m < rows; ++m) {
        const uint16_t *row = R + m * (int64_t)O_K;
        for (int h = 0; h < O_H; ++h) {
            double acc = 0.0;
            for (int i = 0; i < O_HC; ++i)
                acc += pre[m * O_HC + i] * oracle_bf16_to_double(row[i * O_H + h]);
            y[h] = round_y ? oracle_bf16_to_double(oracle_double_to_bf16(acc)) : acc;
        }
        double ss = 0.0;
        for (int h = 0; h < O_H; ++h)
            ss += y[h] * y[h];
        double rn = 1.0 / sqrt(ss / (double)O_H + norm_eps);
        for (int h = 0; h < O_H; ++h)
            x_norm[m * (int64_t)O_H + h] =
                oracle_double_to_bf16(y[h] * rn * oracle_bf16_to_double(w[h]));
    }
    free(y);
}

/* ---- a5: hc_post ---------------------------------------------------------- */

/* R_out[m, i, h] = bf16( post[m, i] * y[m, h] + sum_j comb[m, j, i] * R[m, j, h] ).
 * post [rows, 4] and comb [rows, 4, 4] are fp32, as the kernels receive them. */
void oracle_post(const uint16_t *R, const uint16_t *y, const float *post, const float *comb,
                 int64_t rows, uint16_t *R_out)
{
    for (int64_t m = 0; m < rows; ++m) {
        const uint16_t *row = R + m * (int64_t)O_K;
        const uint16_t *yr = y + m * (int64_t)O_H;
        for (int i = 0; i < O_HC; ++i) {
            double p = (double)post[m * O_HC + i];
            for (int h = 0; h < O_H; ++h) {
                double acc = p * oracle_bf16_to_double(yr[h]);
                for (int j = 0; j < O_HC; ++j)
                    acc += (double)comb[m * 16 + j * 4 + i] *
                           oracle_bf16_to_double(row[j * O_H + h]);
                R_out[m * (int64_t)O_K + i * O_H + h] = oracle_double_to_bf16(acc);
            }
        }
    }
}

/* ---- whole pre pass ------------------------------------------------------- */

/* a1..a4 for rows of R.  Any of the double outputs may be NULL except pre
 * (needed by the combine); post and comb are always produced. */
void oracle_pre(const uint16_t *R, int64_t rows, const float *fn, const float *scale,
                const float *base, const uint16_t *w, double rms_eps, double pre_eps,
                double sink_eps, double norm_eps, double post_mult, int iters,
                double *mix, double *logits, double *pre, double *post, double *comb,
                uint16_t *x_norm)
{
    double *mix_buf = mix ? mix : (double *)malloc(sizeof(double) * O_MIX * (size_t)(rows ? rows : 1));
    oracle_stats(R, rows, fn, rms_eps, mix_buf, NULL);
    oracle_split_sinkhorn(mix_buf, rows, scale, base, pre_eps, sink_eps, post_mult, iters,
                          logits, pre, post, comb);
    if (x_norm)
        oracle_combine_norm(R, rows, pre, w, norm_eps, 0, x_norm);
    if (!mix)
        free(mix_buf);
}

/* ---- hc_head: the final collapse of the streams --------------------------- */

/* For each row m, with x = R[m] flattened stream-major:
 *   rsq       = 1 / sqrt( (sum_k x_k^2) / 20480 + norm_eps )
 *   mix[m, c] = rsq * sum_k x_k * fn[c, k]                 (c = 0..3)
 *   pre[m, i] = sigmoid( mix[m, i] * scale[0] + base[i] ) + hc_eps
 *   y[m, h]   = bf16( sum_i pre[m, i] * R[m, i, h] )
 * fn is [4, 20480] fp32, base [4], scale [1].  mix and pre may be NULL. */
void oracle_hc_head(const uint16_t *R, int64_t rows, const float *fn, const float *scale,
                    const float *base, double norm_eps, double hc_eps, double *mix,
                    double *pre, uint16_t *y)
{
    double *x = (double *)malloc(sizeof(double) * O_K);
    for (int64_t m = 0; m < rows; ++m) {
        const uint16_t *row = R + m * (int64_t)O_K;
        double ss = 0.0;
        for (int k = 0; k < O_K; ++k) {
            x[k] = oracle_bf16_to_double(row[k]);
            ss += x[k] * x[k];
        }
        double r = 1.0 / sqrt(ss / (double)O_K + norm_eps);
        double p[O_HC];
        for (int c = 0; c < O_HC; ++c) {
            const float *f = fn + (int64_t)c * O_K;
            double dot = 0.0;
            for (int k = 0; k < O_K; ++k)
                dot += x[k] * (double)f[k];
            double mx = dot * r;
            if (mix)
                mix[m * O_HC + c] = mx;
            p[c] = sigmoid(mx * (double)scale[0] + (double)base[c]) + hc_eps;
            if (pre)
                pre[m * O_HC + c] = p[c];
        }
        for (int h = 0; h < O_H; ++h) {
            double acc = 0.0;
            for (int i = 0; i < O_HC; ++i)
                acc += p[i] * x[i * O_H + h];
            y[m * (int64_t)O_H + h] = oracle_double_to_bf16(acc);
        }
    }
    free(x);
}

/* ---- MXFP8: E4M3 codes with ue8m0 block scales ----------------------------- */

/* E4M3 (OCP 8-bit float: sign, 4 exponent bits with bias 7, 3 mantissa bits,
 * no infinities, exponent 15 with mantissa 7 is NaN).  A normal code is
 * (1 + m/8) * 2^(E-7), E = 1..15; a subnormal (m/8) * 2^-6.  The largest
 * finite value is 448 (0x7E).  Rounds a finite double to nearest, ties to the
 * even mantissa, and saturates to 448. */
static uint8_t e4m3_from_double(double v)
{
    uint8_t sign = signbit(v) ? 0x80 : 0;
    if (isnan(v))
        return sign | 0x7F;
    double a = fabs(v);
    int q;                        /* quantum exponent of a's binade */
    if (a >= ldexp(1.0, -6)) {
        int e;
        (void)frexp(a, &e);       /* a in [2^(e-1), 2^e) */
        q = (e - 1) - 3;
    } else {
        q = -9;                   /* subnormal quantum */
    }
    double t = ldexp(nearbyint(ldexp(a, -q)), q);   /* exact scaling, one rounding */
    if (t > 448.0)
        t = 448.0;
    if (t == 0.0)
        return sign;
    if (t < ldexp(1.0, -6))
        return sign | (uint8_t)(t * 512.0);         /* subnormal mantissa t / 2^-9 */
    int e;
    double f = frexp(t, &e);      /* t = (2f) * 2^(e-1), 2f in [1, 2) */
    int E = (e - 1) + 7;
    int m = (int)((2.0 * f - 1.0) * 8.0);           /* exact: t has 4 significant bits */
    return sign | (uint8_t)(E << 3) | (uint8_t)m;
}

/* x [rows, cols] bf16 bits, cols a multiple of 32 (finite values).  For each
 * row m and block b of 32 columns:
 *   amax  = max |x[m, 32b .. 32b+31]|
 *   e     = floor(log2 amax) - 8, clamped to [-127, 127]; e = -127 when amax = 0
 *   s[m, b] = e + 127                              (ue8m0 code of 2^e)
 *   q[m, k] = E4M3( x[m, k] / 2^e )                (nearest-even, saturating)
 * q is [rows, cols], s is [rows, cols/32] (the linear layout). */
void oracle_mxfp8_quantize(const uint16_t *x, int64_t rows, int64_t cols, uint8_t *q,
                           uint8_t *s)
{
    const int64_t nb = cols / 32;
    for (int64_t m = 0; m < rows; ++m) {
        for (int64_t b = 0; b < nb; ++b) {
            const uint16_t *blk = x + m * cols + 32 * b;
            double amax = 0.0;
            for (int k = 0; k < 32; ++k) {
                double a = fabs(oracle_bf16_to_double(blk[k]));
                if (a > amax)
                    amax = a;
            }
            int e = -127;
            if (amax > 0.0) {
                int ex;
                (void)frexp(amax, &ex);             /* amax in [2^(ex-1), 2^ex) */
                e = (ex - 1) - 8;
                if (e < -127)
                    e = -127;
                if (e > 127)
                    e = 127;
            }
            s[m * nb + b] = (uint8_t)(e + 127);
            for (int k = 0; k < 32; ++k)
                q[m * cols + 32 * b + k] =
                    e4m3_from_double(ldexp(oracle_bf16_to_double(blk[k]), -e));
        }
    }
}

/* The 128x4 tiled scale layout (prefill_sp.py, swizzle_128x4): s [rows,
 * groups] (groups a multiple of 4) -> out of ceil(rows/128)*128*groups bytes.
 * Rows are padded to a multiple of 128 with zero scales; tile (m/128, g/4) is
 * the (m/128 * groups/4 + g/4)-th run of 512 bytes, and inside it the byte
 * of (m, g) sits at [m%32][(m%128)/32][g%4]. */
void oracle_swizzle_128x4(const uint8_t *s, int64_t rows, int64_t groups, uint8_t *out)
{
    const int64_t tm = (rows + 127) / 128, tg = groups / 4;
    memset(out, 0, (size_t)(tm * 128 * groups));
    for (int64_t m = 0; m < rows; ++m)
        for (int64_t g = 0; g < groups; ++g) {
            int64_t tile = (m / 128) * tg + g / 4;
            int64_t inner = (m % 32) * 16 + ((m % 128) / 32) * 4 + g % 4;
            out[tile * 512 + inner] = s[m * groups + g];
        }
}
