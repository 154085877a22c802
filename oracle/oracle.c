/*
 * oracle.c -- plain, slow CPU oracle for the fused adaLN norm+modulate row
 * kernels.  TEST INFRASTRUCTURE ONLY: the tests, the smoke check and the
 * bench's CPU-baseline leg load it; the product path never does.  It shares
 * no code, header, table or helper with the CUDA library.
 *
 * Build: gcc -O2 -std=c11 -ffp-contract=off -fno-fast-math -shared -fPIC.
 * Contraction must stay off: every "rn(a op b)" below is meant as one IEEE
 * binary32 operation rounded to nearest-even, never fused into an FMA.
 *
 * Sources (the pages are web reports on the sglang diffusion kernels):
 *  - "SGLang diffusion fused-op package guide", section "Norm + scale/shift
 *    (adaLN)": the canonical RMS fragment order (thread tx owns columns
 *    8*TPR*b + 8*tx + v, v fastest then b, one ordered fadd chain per
 *    thread, squares rounded separately), the butterfly fold over offsets
 *    1,2,4,8,16 (= the adjacent-pair tree), the aten modulate chain that
 *    rounds to bf16 after 1+scale, after the product and after +shift, and
 *    the residual variant round(gate*update) then round(residual+that).
 *  - "PR #33854 report" (ERNIE-Image), key source excerpt: pass 1 sum of
 *    squares, the WPR==2 combination w0+w1, s/D + eps, pass 2
 *    (bf16)(x*rstd*w), bf16(1+scale), bf16(y*that), store of prod+shift.
 *  - "PR #34126 report" (FLUX.1), motivation section: LayerNorm with
 *    no affine as per-element Welford and a count-weighted combine; the
 *    guide's bit-exact kernel section adds "128-thread Welford, guarded
 *    reciprocal, shfl.down fold order".
 *  - the guide's list of fused producers: FLUX.2's LayerNorm, adaLN
 *    modulate and static FP8 quantisation folded into one kernel.
 *  - "PR #37123 report" (Qwen-Image), implementation section 3: one
 *    epilogue doing per-head warp-reduced RMSNorm with weight, interleaved
 *    RoPE from an fp32 cos/sin cache for Q and K, a copy for V, written to
 *    joint buffers in [text, image] order.
 *
 * Readings where the pages are silent or disagree (all listed in the design
 * notes): the reciprocal square root is the defined IEEE pair
 * rn(1/rn(sqrt(v))) instead of the pages' rsqrt.approx; s/D is an IEEE
 * division; more than two warp sums combine by the adjacent-pair tree
 * padded with +0; the LayerNorm Welford multiplies by rn(1/n); the combine's
 * parenthesisation and the 4-warp order (W0+W2)+(W1+W3) are ours; the QK
 * head norm uses 16 logical threads of one 8-element fragment each; the
 * RoPE cache row is [cos_0..cos_63 | sin_0..sin_63].
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

typedef uint16_t bf16_bits;

/* ---------------------------------------------------------------- bf16 */

/* bf16 -> fp32 is exact: the 16 bits become the high half of the word. */
static float widen(bf16_bits h)
{
    uint32_t u = (uint32_t)h << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return f;
}

/* fp32 -> bf16, round to nearest, ties to even, by integer arithmetic on
 * the bit pattern.  Any NaN becomes the quiet NaN 0x7FC0 with its sign. */
static bf16_bits narrow(float f)
{
    uint32_t u;
    memcpy(&u, &f, sizeof u);
    if ((u & 0x7FFFFFFFu) > 0x7F800000u)
        return (bf16_bits)(((u >> 16) & 0x8000u) | 0x7FC0u);
    u += 0x7FFFu + ((u >> 16) & 1u);
    return (bf16_bits)(u >> 16);
}

/* bf(f): the fp32 value of the bf16 nearest to f. */
static float bf(float f) { return widen(narrow(f)); }

/* One IEEE binary32 operation each (contraction is off for this file). */
static float rn_add(float a, float b) { return a + b; }
static float rn_sub(float a, float b) { return a - b; }
static float rn_mul(float a, float b) { return a * b; }
static float rn_div(float a, float b) { return a / b; }

/* The defined reciprocal square root: two correctly rounded operations. */
static float defined_rsqrt(float v) { return rn_div(1.0f, sqrtf(v)); }

/* ----------------------------------------------------------- modulate */

/* y = bf(rn(bf(n * bf(rn(1 + scale))) + shift)); n is already bf16.  The
 * product of two bf16 values is exact in fp32, so bf() rounds it once. */
static bf16_bits modulate(float n, float scale, float shift)
{
    float one_plus = bf(rn_add(1.0f, scale));
    float p = bf(rn_mul(n, one_plus));
    return narrow(rn_add(p, shift));
}

/* ------------------------------------------------------------ RMSNorm */

/* Canonical sum of squares of one row of D = 64*TPR values.
 * Logical thread tx in [0,TPR) owns columns 8*TPR*b + 8*tx + v, b,v in
 * [0,8), and sums rn(x*x) into one sequential chain with v fastest.  Each
 * group of 32 consecutive threads (a warp) folds its partials by the
 * adjacent-pair tree; the warp sums fold by the same tree, padded with +0
 * up to a power of two (two warps: w0 + w1).  Threads past TPR in the last
 * warp contribute +0. */
static float rms_sum_of_squares(const float *x, int64_t D)
{
    int64_t tpr = D / 64;
    int64_t nwarps = (tpr + 31) / 32;
    int64_t npow = 1;
    while (npow < nwarps)
        npow *= 2;
    float *wsum = (float *)calloc((size_t)npow, sizeof(float));
    for (int64_t w = 0; w < nwarps; ++w) {
        float lane[32];
        for (int l = 0; l < 32; ++l) {
            int64_t tx = 32 * w + l;
            float acc = 0.0f;
            if (tx < tpr)
                for (int b = 0; b < 8; ++b)
                    for (int v = 0; v < 8; ++v) {
                        float xv = x[8 * tpr * b + 8 * tx + v];
                        acc = rn_add(acc, rn_mul(xv, xv));
                    }
            lane[l] = acc;
        }
        for (int off = 1; off < 32; off *= 2)
            for (int i = 0; i < 32; i += 2 * off)
                lane[i] = rn_add(lane[i], lane[i + off]);
        wsum[w] = lane[0];
    }
    for (int64_t off = 1; off < npow; off *= 2)
        for (int64_t i = 0; i < npow; i += 2 * off)
            wsum[i] = rn_add(wsum[i], wsum[i + off]);
    float s = wsum[0];
    free(wsum);
    return s;
}

/* Normalise + modulate one row given its widened values. */
static void rms_row(const float *xrow, const bf16_bits *w, const bf16_bits *scale,
                    const bf16_bits *shift, bf16_bits *y, int64_t D, float eps,
                    float *stats)
{
    float s = rms_sum_of_squares(xrow, D);
    float mean_sq = rn_div(s, (float)D);
    float rstd = defined_rsqrt(rn_add(mean_sq, eps));
    for (int64_t j = 0; j < D; ++j) {
        float t = rn_mul(xrow[j], rstd);
        float n = w ? bf(rn_mul(t, widen(w[j]))) : bf(t);
        y[j] = modulate(n, widen(scale[j]), widen(shift[j]));
    }
    if (stats) {
        stats[0] = s;
        stats[1] = rstd;
    }
}

/* y = bf16(rms(x) (*w) * (1+scale) + shift) for x [B,T,D]; scale/shift
 * rows of batch b start at b*vs.  stats (nullable): per row {s, rstd}.
 * Requires D % 64 == 0 (the CUDA library further requires D % 2048 == 0). */
void oracle_rms_modulate(const bf16_bits *x, const bf16_bits *weight,
                         const bf16_bits *scale, const bf16_bits *shift, int64_t vs,
                         bf16_bits *y, int64_t B, int64_t T, int64_t D, float eps,
                         float *stats)
{
    float *xrow = (float *)malloc((size_t)D * sizeof(float));
    for (int64_t r = 0; r < B * T; ++r) {
        int64_t b = r / T;
        for (int64_t j = 0; j < D; ++j)
            xrow[j] = widen(x[r * D + j]);
        rms_row(xrow, weight, scale + b * vs, shift + b * vs, y + r * D, D, eps,
                stats ? stats + 2 * r : NULL);
    }
    free(xrow);
}

/* Gated residual: r' = bf(rn(r + bf(rn(gate*h)))), stored to r_out, then the
 * RMS row above on r'.  r_out may equal r (each element is read first). */
void oracle_gated_rms_modulate(const bf16_bits *r, const bf16_bits *h,
                               const bf16_bits *gate, const bf16_bits *weight,
                               const bf16_bits *scale, const bf16_bits *shift, int64_t vs,
                               bf16_bits *r_out, bf16_bits *y, int64_t B, int64_t T,
                               int64_t D, float eps, float *stats)
{
    float *xrow = (float *)malloc((size_t)D * sizeof(float));
    for (int64_t row = 0; row < B * T; ++row) {
        int64_t b = row / T;
        for (int64_t j = 0; j < D; ++j) {
            float gh = bf(rn_mul(widen(gate[b * vs + j]), widen(h[row * D + j])));
            bf16_bits rp = narrow(rn_add(widen(r[row * D + j]), gh));
            r_out[row * D + j] = rp;
            xrow[j] = widen(rp);
        }
        rms_row(xrow, weight, scale + b * vs, shift + b * vs, y + row * D, D, eps,
                stats ? stats + 2 * row : NULL);
    }
    free(xrow);
}

/* ---------------------------------------------------------- LayerNorm */

typedef struct {
    float n, mean, m2;
} welford;

/* Count-weighted combine of two partial states (Chan, Golub, LeVeque),
 * A being the lower lane or warp.  An empty side returns the other. */
static welford welford_combine(welford A, welford B)
{
    if (B.n == 0.0f)
        return A;
    if (A.n == 0.0f)
        return B;
    welford o;
    o.n = rn_add(A.n, B.n);
    float c = rn_div(B.n, o.n);
    float delta = rn_sub(B.mean, A.mean);
    o.mean = rn_add(A.mean, rn_mul(delta, c));
    o.m2 = rn_add(rn_add(A.m2, B.m2), rn_mul(rn_mul(rn_mul(delta, delta), A.n), c));
    return o;
}

/* 128 logical threads; thread t owns the 8-element fragments starting at
 * column 8*(t + 128*k), k = 0,1,... while < D, visited in k order, v = 0..7
 * inside.  Per element (Welford): n += 1; d = x - mean;
 * mean += d*rn(1/n); m2 += d*(x - mean).  Each warp of 32 threads folds by
 * the shfl.down order (offsets 16,8,4,2,1: lane i takes i (+) i+off); the
 * four warp results fold the same way with offsets 2,1. */
static welford ln_statistics(const float *x, int64_t D)
{
    welford lane[128];
    for (int t = 0; t < 128; ++t) {
        welford s = {0.0f, 0.0f, 0.0f};
        for (int64_t base = 8 * (int64_t)t; base < D; base += 8 * 128)
            for (int v = 0; v < 8; ++v) {
                float xv = x[base + v];
                s.n = rn_add(s.n, 1.0f);
                float inv_n = rn_div(1.0f, s.n);
                float d = rn_sub(xv, s.mean);
                s.mean = rn_add(s.mean, rn_mul(d, inv_n));
                float d2 = rn_sub(xv, s.mean);
                s.m2 = rn_add(s.m2, rn_mul(d, d2));
            }
        lane[t] = s;
    }
    welford warp[4];
    for (int w = 0; w < 4; ++w) {
        welford *l = lane + 32 * w;
        for (int off = 16; off >= 1; off /= 2)
            for (int i = 0; i < off; ++i)
                l[i] = welford_combine(l[i], l[i + off]);
        warp[w] = l[0];
    }
    for (int off = 2; off >= 1; off /= 2)
        for (int i = 0; i < off; ++i)
            warp[i] = welford_combine(warp[i], warp[i + off]);
    return warp[0];
}

/* One LayerNorm + modulate row: n = bf(rn(rn(x - mean) * rstd)),
 * rstd = rn(1/rn(sqrt(rn(rn(m2/D) + eps)))), y = modulate(n, scale, shift).
 * stats (nullable): {mean, m2, rstd}. */
static void ln_row(const float *xrow, const bf16_bits *scale, const bf16_bits *shift,
                   bf16_bits *y, int64_t D, float eps, float *stats)
{
    welford st = ln_statistics(xrow, D);
    float var = rn_div(st.m2, (float)D);
    float rstd = defined_rsqrt(rn_add(var, eps));
    for (int64_t j = 0; j < D; ++j) {
        float n = bf(rn_mul(rn_sub(xrow[j], st.mean), rstd));
        y[j] = modulate(n, widen(scale[j]), widen(shift[j]));
    }
    if (stats) {
        stats[0] = st.mean;
        stats[1] = st.m2;
        stats[2] = rstd;
    }
}

/* y = bf16(LN(x) * (1+scale) + shift), LayerNorm without affine.
 * stats (nullable): per row {mean, m2, rstd}.  Requires D % 8 == 0. */
void oracle_ln_modulate(const bf16_bits *x, const bf16_bits *scale, const bf16_bits *shift,
                        int64_t vs, bf16_bits *y, int64_t B, int64_t T, int64_t D, float eps,
                        float *stats)
{
    float *xrow = (float *)malloc((size_t)D * sizeof(float));
    for (int64_t r = 0; r < B * T; ++r) {
        int64_t b = r / T;
        for (int64_t j = 0; j < D; ++j)
            xrow[j] = widen(x[r * D + j]);
        ln_row(xrow, scale + b * vs, shift + b * vs, y + r * D, D, eps,
               stats ? stats + 3 * r : NULL);
    }
    free(xrow);
}

/* The gated residual form with LayerNorm: r' = bf(rn(r + bf(rn(gate * h))))
 * is stored, then y = the LayerNorm + modulate row of r'.  The guide's
 * residual variant (round(gate*update), then round(residual + that), the
 * rounded result fed to the same faithful norm) with the LayerNorm of the
 * FLUX pages in place of RMSNorm.  gate, scale, shift share vs. */
void oracle_gated_ln_modulate(const bf16_bits *r, const bf16_bits *h, const bf16_bits *gate,
                              const bf16_bits *scale, const bf16_bits *shift, int64_t vs,
                              bf16_bits *r_out, bf16_bits *y, int64_t B, int64_t T, int64_t D,
                              float eps, float *stats)
{
    float *xrow = (float *)malloc((size_t)D * sizeof(float));
    for (int64_t row = 0; row < B * T; ++row) {
        int64_t b = row / T;
        for (int64_t j = 0; j < D; ++j) {
            float gh = bf(rn_mul(widen(gate[b * vs + j]), widen(h[row * D + j])));
            bf16_bits rp = narrow(rn_add(widen(r[row * D + j]), gh));
            r_out[row * D + j] = rp;
            xrow[j] = widen(rp);
        }
        ln_row(xrow, scale + b * vs, shift + b * vs, y + row * D, D, eps,
               stats ? stats + 3 * row : NULL);
    }
    free(xrow);
}

/* ------------------------------------------------- QK norm + RoPE + V */

/* RMS of one head of hd values (hd = 128 or 64): hd/8 logical threads,
 * thread l owns columns 8l..8l+7 as one chain; the partials fold by the
 * adjacent-pair tree. */
static float head_rstd(const float *x, int hd, float eps)
{
    float lane[16];
    const int L = hd / 8;
    for (int l = 0; l < L; ++l) {
        float acc = 0.0f;
        for (int v = 0; v < 8; ++v)
            acc = rn_add(acc, rn_mul(x[8 * l + v], x[8 * l + v]));
        lane[l] = acc;
    }
    for (int off = 1; off < L; off *= 2)
        for (int i = 0; i < L; i += 2 * off)
            lane[i] = rn_add(lane[i], lane[i + off]);
    return defined_rsqrt(rn_add(rn_div(lane[0], (float)hd), eps));
}

/* Normalise one head with weight w, then rotate by the cos/sin of cache row
 * rope ([cos_0..cos_{hd/2-1} | sin_0..sin_{hd/2-1}], fp32): interleaved
 * pairs (2i, 2i+1), or with neox != 0 the halves' pairs (i, i + hd/2). */
static float qk_head(const bf16_bits *src, const bf16_bits *w, const float *rope, int hd,
                     int neox, float eps, bf16_bits *dst)
{
    float x[128], n[128];
    const int half = hd / 2;
    for (int j = 0; j < hd; ++j)
        x[j] = widen(src[j]);
    float rstd = head_rstd(x, hd, eps);
    for (int j = 0; j < hd; ++j)
        n[j] = bf(rn_mul(rn_mul(x[j], rstd), widen(w[j])));
    for (int i = 0; i < half; ++i) {
        const float c = rope[i], s = rope[half + i];
        const int ia = neox ? i : 2 * i, ib = neox ? i + half : 2 * i + 1;
        const float a = n[ia], b = n[ib];
        dst[ia] = narrow(rn_sub(rn_mul(a, c), rn_mul(b, s)));
        dst[ib] = narrow(rn_add(rn_mul(a, s), rn_mul(b, c)));
    }
    return rstd;
}

static void qk_stream(const bf16_bits *q, const bf16_bits *k, const bf16_bits *v, int64_t T,
                      int64_t stride, int64_t H, int hd, int neox, const bf16_bits *wq,
                      const bf16_bits *wk, const float *rope, float eps, int64_t out_row0,
                      bf16_bits *q_out, bf16_bits *k_out, bf16_bits *v_out, float *rstd_out)
{
    for (int64_t t = 0; t < T; ++t) {
        int64_t orow = out_row0 + t;
        for (int64_t h = 0; h < H; ++h) {
            int64_t src = t * stride + h * hd;
            int64_t dst = (orow * H + h) * hd;
            float rq = qk_head(q + src, wq, rope + t * hd, hd, neox, eps, q_out + dst);
            float rk = qk_head(k + src, wk, rope + t * hd, hd, neox, eps, k_out + dst);
            memcpy(v_out + dst, v + src, (size_t)hd * sizeof(bf16_bits));
            if (rstd_out) {
                rstd_out[(orow * 2 + 0) * H + h] = rq;
                rstd_out[(orow * 2 + 1) * H + h] = rk;
            }
        }
    }
}

/* Q/K: per-head RMSNorm with weight then RoPE; V: copy.  Inputs are
 * row-strided views (row stride in elements, heads contiguous at hd);
 * outputs are [T_txt + T_img, H, hd], text rows first.  hd is 128 or 64;
 * neox selects the rotation of halves instead of interleaved pairs (the
 * interleaved form is the Qwen epilogue's is_neox=False).  rstd_out
 * (nullable): [T_txt + T_img, 2 (q,k), H]. */
void oracle_qk_norm_rope(const bf16_bits *q_txt, const bf16_bits *k_txt, const bf16_bits *v_txt,
                         int64_t T_txt, int64_t txt_stride, const bf16_bits *q_img,
                         const bf16_bits *k_img, const bf16_bits *v_img, int64_t T_img,
                         int64_t img_stride, int64_t H, int hd, int neox,
                         const bf16_bits *wq_txt, const bf16_bits *wk_txt,
                         const bf16_bits *wq_img, const bf16_bits *wk_img,
                         const float *rope_txt, const float *rope_img, float eps_txt,
                         float eps_img, bf16_bits *q_out, bf16_bits *k_out, bf16_bits *v_out,
                         float *rstd_out)
{
    qk_stream(q_txt, k_txt, v_txt, T_txt, txt_stride, H, hd, neox, wq_txt, wk_txt, rope_txt,
              eps_txt, 0, q_out, k_out, v_out, rstd_out);
    qk_stream(q_img, k_img, v_img, T_img, img_stride, H, hd, neox, wq_img, wk_img, rope_img,
              eps_img, T_txt, q_out, k_out, v_out, rstd_out);
}

/* The Qwen epilogue: head_dim 128, interleaved pairs. */
void oracle_qk_norm_rope_epilogue(const bf16_bits *q_txt, const bf16_bits *k_txt,
                                  const bf16_bits *v_txt, int64_t T_txt, int64_t txt_stride,
                                  const bf16_bits *q_img, const bf16_bits *k_img,
                                  const bf16_bits *v_img, int64_t T_img, int64_t img_stride,
                                  int64_t H, const bf16_bits *wq_txt, const bf16_bits *wk_txt,
                                  const bf16_bits *wq_img, const bf16_bits *wk_img,
                                  const float *rope_txt, const float *rope_img, float eps_txt,
                                  float eps_img, bf16_bits *q_out, bf16_bits *k_out,
                                  bf16_bits *v_out, float *rstd_out)
{
    oracle_qk_norm_rope(q_txt, k_txt, v_txt, T_txt, txt_stride, q_img, k_img, v_img, T_img,
                        img_stride, H, 128, 0, wq_txt, wk_txt, wq_img, wk_img, rope_txt,
                        rope_img, eps_txt, eps_img, q_out, k_out, v_out, rstd_out);
}

/* ------------------------------------- residual gating, transposed layout */

/* The residual stream in the [B, hidden, tokens] layout: r, r_out are
 * [B, D, T], the update h is [B, T, D] (logical row-major), gate [B, D]
 * with batch stride vs:  r_out[b,d,t] = bf(rn(r[b,d,t] + bf(rn(gate[b,d] *
 * h[b,t,d])))).  The guide's residual-gating variant ("Norm variants /
 * residual gating"): the transposed dense path reads the update in logical
 * row-major order and keeps the residual reads and output writes in their
 * [B, hidden, tokens] layout. */
void oracle_gated_residual_transposed(const bf16_bits *r, const bf16_bits *h,
                                      const bf16_bits *gate, int64_t vs, bf16_bits *r_out,
                                      int64_t B, int64_t T, int64_t D)
{
    for (int64_t b = 0; b < B; ++b)
        for (int64_t d = 0; d < D; ++d) {
            const float g = widen(gate[b * vs + d]);
            for (int64_t t = 0; t < T; ++t) {
                const int64_t i = (b * D + d) * T + t;
                const float gh = bf(rn_mul(g, widen(h[(b * T + t) * D + d])));
                r_out[i] = narrow(rn_add(widen(r[i]), gh));
            }
        }
}

/* ------------------------------------------- LayerNorm + modulate + FP8 */

/* fp32 -> FP8 E4M3 (OCP "e4m3fn": 1 sign, 4 exponent bits with bias 7, 3
 * mantissa bits; no infinities; S.1111.111 is NaN; largest finite 448),
 * rounded to nearest with ties to even and saturated: a finite or infinite
 * value of magnitude >= 448 becomes +-448.  Any NaN becomes 0x7F.
 * Written from the format's definition: the representable values of the
 * binade of |v| (or the subnormal range below 2^-6) are the multiples of
 * one power-of-two quantum, so |v| / quantum is exact and rintf (round half
 * to even in the default rounding mode) picks the nearest one. */
static uint8_t e4m3_satfinite(float v)
{
    if (isnan(v)) return 0x7F;
    const uint8_t sign = signbit(v) ? 0x80 : 0x00;
    const float a = fabsf(v);
    if (a >= 448.0f) return (uint8_t)(sign | 0x7E);
    int e = 0;
    (void)frexpf(a, &e); /* a = m * 2^e with m in [0.5, 1); floor(log2 a) = e - 1 */
    int ex = e - 1;
    if (a == 0.0f || ex < -6) ex = -6; /* subnormal range: quantum 2^-9 */
    const float quantum = ldexpf(1.0f, ex - 3);
    const float k = rintf(a / quantum);
    const float r = k * quantum; /* exact */
    if (r == 0.0f) return sign;
    if (r < ldexpf(1.0f, -6)) return (uint8_t)(sign | (uint8_t)k); /* subnormal: k/8 * 2^-6 */
    (void)frexpf(r, &e);
    const int biased = (e - 1) + 7;
    const int frac = (int)(ldexpf(r, -(e - 1)) * 8.0f) - 8; /* r / 2^(e-1) = 1 + frac/8 */
    return (uint8_t)(sign | (uint8_t)((biased << 3) | frac));
}

/* q = e4m3(rn(y * inv_s)) per element, y the bf16 result of
 * oracle_ln_modulate, inv_s = rn(1 / qscale) for a static (per-tensor)
 * quantisation scale qscale > 0.  "SGLang diffusion fused-op package
 * guide", list of fused producers: FLUX.2's LayerNorm, adaLN modulate and
 * static FP8 quantisation in one kernel.  The reciprocal multiply, the
 * E4M3 format and the saturation are this library's readings. */
void oracle_ln_modulate_fp8(const bf16_bits *x, const bf16_bits *scale, const bf16_bits *shift,
                            int64_t vs, float qscale, uint8_t *q, int64_t B, int64_t T,
                            int64_t D, float eps)
{
    const float inv_s = rn_div(1.0f, qscale);
    bf16_bits *y = (bf16_bits *)malloc((size_t)(B * T * D) * sizeof(bf16_bits) + 1);
    oracle_ln_modulate(x, scale, shift, vs, y, B, T, D, eps, NULL);
    for (int64_t i = 0; i < B * T * D; ++i)
        q[i] = e4m3_satfinite(rn_mul(widen(y[i]), inv_s));
    free(y);
}

/* ------------------------------------------------------ exported helpers */

/* The oracle's own fp32 -> E4M3 conversion, exposed for the tests. */
void oracle_fp8_e4m3(const float *in, uint8_t *out, int64_t n)
{
    for (int64_t i = 0; i < n; ++i)
        out[i] = e4m3_satfinite(in[i]);
}


/* The oracle's own fp32 -> bf16 rounding, exposed so that tests can pin it
 * against an independent formulation. */
void oracle_round_bf16(const float *in, bf16_bits *out, int64_t n)
{
    for (int64_t i = 0; i < n; ++i)
        out[i] = narrow(in[i]);
}
