/*
 * dan.h -- C ABI of the GB300 (sm_103a) fused adaLN norm+modulate kernels.
 *
 * Eight operations, each a single kernel launch on the caller's stream:
 *
 *   dan_ln_modulate         y = bf16(LayerNorm(x) * (1 + scale) + shift)
 *   dan_ln_modulate_fp8     q = e4m3(y * rn(1/qscale)), y as dan_ln_modulate
 *   dan_gated_ln_modulate   r' = bf16(r + bf16(gate * h)); y = ln_modulate(r')
 *   dan_gated_residual_transposed  r' = bf16(r + bf16(gate * h)) with the
 *                           residual in the [B, hidden, tokens] layout
 *   dan_rms_modulate        y = bf16(RMSNorm(x) [* w] * (1 + scale) + shift)
 *   dan_gated_rms_modulate  r' = bf16(r + bf16(gate * h)); y = rms_modulate(r')
 *   dan_qk_norm_rope_epilogue  per-head RMSNorm + interleaved RoPE of Q and K,
 *                           copy of V, into joint [text, image] buffers
 *   dan_qk_norm_rope_neox_epilogue  the same with the neox rotation of halves
 *
 * The operations are the ones described on these pages:
 *  - "SGLang diffusion fused-op package guide", section "Norm + scale/shift
 *    (adaLN)": canonical RMS fragment order and butterfly fold, the aten
 *    modulate chain (bf16 rounding after 1+scale, after the product and
 *    after +shift), and the residual variant (round(gate*update), then
 *    round(residual + that)).
 *  - "PR #33854 report" (ERNIE-Image bit-exact RMSNorm+scale/shift), key
 *    source excerpt: one row per program, optional norm weight, gated form
 *    that also returns the updated residual.
 *  - "PR #34126 report" (FLUX.1 fused LayerNorm+modulate), motivation
 *    section: LayerNorm without affine by Welford; the guard hidden % 4 == 0
 *    and hidden <= 8192 (related-work section).
 *  - "PR #37123 report" (Qwen-Image FP8 QKV + Blackwell epilogue),
 *    implementation section 3: guards bf16, batch 1, head_dim 128, aligned
 *    data pointers, head stride 128, Q/K/V sharing one layout; RMSNorm with
 *    weight per head, interleaved RoPE from fp32 cos/sin rows, V copied,
 *    outputs in [text, image] order.
 *
 * Numerics.  Every result is defined bit for bit: fp32 operations rounded to
 * nearest-even one at a time (never fused into FMA), bf16 rounding to
 * nearest-even at the boundaries above, a defined reciprocal square root
 * rstd = rn(1 / rn(sqrt(v))), and a fixed reduction order per row that does
 * not depend on B, T, the grid or the launch.  A row's output bits are
 * therefore the same whatever batch it is computed in.  NaN results are some
 * quiet NaN (payload unspecified).
 *
 * Conventions for every entry point.
 *  - bf16 tensors are passed as raw 16-bit patterns (dan_bf16).  All tensor
 *    pointers are DEVICE pointers owned by the caller; the library never
 *    allocates, frees or synchronises.  `stream` is a cudaStream_t (NULL =
 *    the legacy default stream); the launch is asynchronous on it.
 *  - Launches allow programmatic dependent launch: a kernel may begin while
 *    the previous kernel in the stream is finishing.  Until that kernel has
 *    completed it only sets up its shared memory and hints its first inputs
 *    into L2 (a hint returns no data); it reads inputs only after waiting
 *    for that completion, so stream order holds exactly.
 *  - Row tensors [B, T, D] are contiguous, row r = b*T + t.  Per-batch
 *    vectors (scale, shift, gate) are rows of a [B, D] matrix whose batch
 *    stride is `vec_bstride` elements (>= D, a multiple of 8), e.g. chunks
 *    of one adaLN embedding row; `weight` is one contiguous [D] vector.
 *  - Every pointer must be 16-byte aligned (DAN_EALIGN otherwise).
 *  - Outputs may not overlap any input or each other (DAN_EALIAS), except
 *    the exact in-place forms named below.
 *  - B * T == 0 (or T_txt + T_img == 0) launches nothing and returns DAN_OK.
 *  - Invalid arguments return a status without launching and without side
 *    effects.  DAN_ECUDA means the launch itself failed; the CUDA error is
 *    left for the caller to query with cudaGetLastError().
 *  - Each dan_can_use_* takes the same arguments minus the stream, performs
 *    the same validation, launches nothing and touches no memory.
 */
#ifndef DAN_H
#define DAN_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef uint16_t dan_bf16; /* raw bf16 bit pattern */

typedef enum {
    DAN_OK = 0,
    DAN_EINVAL = 1,       /* null pointer, negative size, bad stride, eps < 0 or not finite */
    DAN_EUNSUPPORTED = 2, /* D or head_dim outside the supported set */
    DAN_EALIGN = 3,       /* a pointer or stride breaks 16-byte alignment */
    DAN_EALIAS = 4,       /* an output overlaps an input or another output */
    DAN_ECUDA = 5         /* the kernel launch failed */
} dan_status;

/* Human-readable name of a status code (static string, never NULL). */
const char *dan_status_string(int status);

/* ------------------------------------------------------ device status
 * The kernels stream rows through shared memory with bulk copies whose
 * completion they wait for on mbarriers.  Every such wait is bounded (about
 * one second); a wait that runs out makes the kernel record a bit in the
 * current device's status word and return, leaving its outputs incomplete:
 *   1 = a warp gave up waiting for a row (or head group) it had requested,
 *   4 = after that, it also gave up waiting for its other copies in flight.
 * (Bit 2 is not used.)
 * dan_get_device_status reads the word of the current device into *status
 * and clears it.  It is synchronous: call it after synchronising the streams
 * the kernels ran on.  Returns DAN_OK, DAN_EINVAL (status NULL) or DAN_ECUDA.
 * The word is static device memory of the library: nothing is allocated. */
int dan_get_device_status(unsigned int *status);

/* Self-test of the bounded wait: launches one warp that waits on an
 * mbarrier nothing completes, for limit_ns nanoseconds (1 .. 2e9), then
 * records status bit 1 and returns.  Lets a test check that a wait that
 * runs out reports through dan_get_device_status and leaves the context
 * usable.  Asynchronous on `stream`. */
int dan_selftest_wait_timeout(unsigned long long limit_ns, void *stream);

/* ------------------------------------------------------------------ RMS
 * y[b,t,:] = bf16(bf16(n * o) + shift) per element, where
 *   n = bf16(rn(x * rstd))             (weight == NULL)
 *   n = bf16(rn(rn(x * rstd) * w))     (weight given, one rounding)
 *   o = bf16(rn(1 + scale))
 *   rstd = rn(1 / rn(sqrt(rn(rn(s / D) + eps))))
 * and s is the sum of rn(x*x) in the canonical order: logical thread tx of
 * TPR = D/64 owns columns 8*TPR*b + 8*tx + v (b, v in 0..7, v fastest) as one
 * sequential fp32 chain; each 32 threads fold by the adjacent-pair tree
 * (butterfly offsets 1,2,4,8,16); the D/2048 warp sums fold by the same tree
 * padded with +0 to a power of two.
 * Supported: D in {2048, 4096, 6144, 8192}.  eps >= 0, finite.
 * In place: y == x is allowed (each row is read completely before it is
 * written). */
int dan_rms_modulate(const dan_bf16 *x, const dan_bf16 *weight, const dan_bf16 *scale,
                     const dan_bf16 *shift, int64_t vec_bstride, dan_bf16 *y, int64_t B,
                     int64_t T, int64_t D, float eps, void *stream);
int dan_can_use_rms_modulate(const dan_bf16 *x, const dan_bf16 *weight, const dan_bf16 *scale,
                             const dan_bf16 *shift, int64_t vec_bstride, const dan_bf16 *y,
                             int64_t B, int64_t T, int64_t D, float eps);

/* RMS + modulate for callers that cannot allocate device memory: code that
 * runs inside a stream capture whose mode forbids allocation calls, or a
 * runtime whose device memory belongs to an allocator of its own (a caching
 * pool that must not see foreign cudaMalloc/cudaFree).  The pages have no
 * counterpart; it is the same kernel and result as dan_rms_modulate (same
 * arguments, validation and output bits).  Its scratch -- one bounded-wait
 * failure record per CTA, kept for the library's own use -- lives in a
 * static device array of 256 records (1 KB) that the library holds on every
 * GPU that loads it until the process exits; no device memory is allocated
 * or freed.  The records are not part of the interface: a caller learns of
 * a failed wait through dan_get_device_status, as for every other call.  The launch uses one CTA per SM (at most the row
 * count); a GPU with more than 256 SMs gets DAN_EUNSUPPORTED.  The first
 * call on a device looks up the array's address (cudaGetSymbolAddress), so
 * make that first call before any stream capture.  Every call shares the
 * array and each CTA clears its record when it starts: calls that overlap
 * on the GPU race on it. */
int dan_rms_modulate_noalloc(const dan_bf16 *x, const dan_bf16 *weight, const dan_bf16 *scale,
                             const dan_bf16 *shift, int64_t vec_bstride, dan_bf16 *y, int64_t B,
                             int64_t T, int64_t D, float eps, void *stream);

/* ------------------------------------------------------------- gated RMS
 * r_out = bf16(rn(r + bf16(rn(gate * h)))) (the updated residual stream),
 * then y = the RMS row above applied to r_out.  gate, scale, shift share
 * vec_bstride.  Supported D as for dan_rms_modulate.
 * In place: r_out == r is allowed; y may not overlap r_out or any input. */
int dan_gated_rms_modulate(const dan_bf16 *r, const dan_bf16 *h, const dan_bf16 *gate,
                           const dan_bf16 *weight, const dan_bf16 *scale, const dan_bf16 *shift,
                           int64_t vec_bstride, dan_bf16 *r_out, dan_bf16 *y, int64_t B,
                           int64_t T, int64_t D, float eps, void *stream);
int dan_can_use_gated_rms_modulate(const dan_bf16 *r, const dan_bf16 *h, const dan_bf16 *gate,
                                   const dan_bf16 *weight, const dan_bf16 *scale,
                                   const dan_bf16 *shift, int64_t vec_bstride,
                                   const dan_bf16 *r_out, const dan_bf16 *y, int64_t B, int64_t T,
                                   int64_t D, float eps);

/* -------------------------------------------------------------- LayerNorm
 * LayerNorm without affine, then the modulate chain:
 *   n = bf16(rn(rn(x - mean) * rstd)),  rstd = rn(1/rn(sqrt(rn(rn(m2/D) + eps))))
 * (population variance).  mean and m2 come from a fixed Welford tree: 128
 * logical threads, thread t owns the 8-element fragments at columns
 * 8*(t + 128k) (k = 0,1,.. while < D); per element n += 1, d = x - mean,
 * mean += d * rn(1/n), m2 += d * (x - mean); partial states combine as
 *   n = nA + nB, c = rn(nB/n), delta = mB - mA, mean = mA + delta*c,
 *   m2 = (m2A + m2B) + ((delta*delta)*nA)*c   (an empty side returns the other),
 * each warp of 32 threads in shfl.down order (offsets 16,8,4,2,1), the four
 * warp results as (W0 + W2) + (W1 + W3).
 * Supported: D % 8 == 0, 8 <= D <= 8192.  In place: y == x is allowed. */
int dan_ln_modulate(const dan_bf16 *x, const dan_bf16 *scale, const dan_bf16 *shift,
                    int64_t vec_bstride, dan_bf16 *y, int64_t B, int64_t T, int64_t D, float eps,
                    void *stream);
int dan_can_use_ln_modulate(const dan_bf16 *x, const dan_bf16 *scale, const dan_bf16 *shift,
                            int64_t vec_bstride, const dan_bf16 *y, int64_t B, int64_t T,
                            int64_t D, float eps);

/* ------------------------------------------------------ gated LayerNorm
 * The residual variant of the guide's "Norm + scale/shift (adaLN)" section
 * (round(gate * update), then round(residual + that), the rounded result
 * fed to the same norm) with the LayerNorm above:
 *   r_out = bf16(rn(r + bf16(rn(gate * h)))),  y = dan_ln_modulate(r_out)
 * bit for bit.  gate, scale, shift share vec_bstride.  Supported D as for
 * dan_ln_modulate.  In place: r_out == r is allowed; y may not overlap
 * r_out or any input. */
int dan_gated_ln_modulate(const dan_bf16 *r, const dan_bf16 *h, const dan_bf16 *gate,
                          const dan_bf16 *scale, const dan_bf16 *shift, int64_t vec_bstride,
                          dan_bf16 *r_out, dan_bf16 *y, int64_t B, int64_t T, int64_t D,
                          float eps, void *stream);
int dan_can_use_gated_ln_modulate(const dan_bf16 *r, const dan_bf16 *h, const dan_bf16 *gate,
                                  const dan_bf16 *scale, const dan_bf16 *shift,
                                  int64_t vec_bstride, const dan_bf16 *r_out, const dan_bf16 *y,
                                  int64_t B, int64_t T, int64_t D, float eps);

/* --------------------------------- residual gating, transposed layout
 * "SGLang diffusion fused-op package guide", norm variants, residual
 * gating: the residual stream r and the output r_out are [B, D, T] (the
 * [B, hidden, tokens] layout), the update h is [B, T, D] (logical
 * row-major), gate [B, D] with batch stride vec_bstride (a multiple of 8,
 * >= D):
 *   r_out[b, d, t] = bf16(rn(r[b, d, t] + bf16(rn(gate[b, d] * h[b, t, d]))))
 * The update is read through shared-memory tiles; the residual reads and
 * r_out writes stay coalesced along the tokens (no transposed copy).
 * Supported: D % 8 == 0, D >= 8, any T.  In place: r_out == r is allowed;
 * r_out may not overlap h or gate.  All pointers 16-byte aligned. */
int dan_gated_residual_transposed(const dan_bf16 *r, const dan_bf16 *h, const dan_bf16 *gate,
                                  int64_t vec_bstride, dan_bf16 *r_out, int64_t B, int64_t T,
                                  int64_t D, void *stream);
int dan_can_use_gated_residual_transposed(const dan_bf16 *r, const dan_bf16 *h,
                                          const dan_bf16 *gate, int64_t vec_bstride,
                                          const dan_bf16 *r_out, int64_t B, int64_t T, int64_t D);

/* ------------------------------------------- LayerNorm + modulate + FP8
 * "SGLang diffusion fused-op package guide", list of fused producers:
 * FLUX.2's LayerNorm, adaLN modulate and static FP8 quantisation folded
 * into one kernel, which feeds an FP8 GEMM.  Per element
 *   q = e4m3(rn(y * rn(1 / qscale)))
 * with y the bf16 result dan_ln_modulate would return (same arguments, same
 * bits) and e4m3 the OCP E4M3 ("e4m3fn") code: round to nearest, ties to
 * even, values of magnitude >= 448 (and infinities) saturated to +-448, NaN
 * to a NaN code.  qscale is the static per-tensor scale (finite, > 0);
 * rn(1/qscale) is one IEEE division on the host.  q is [B, T, D] bytes,
 * contiguous, 16-byte aligned, and may not overlap any input (no in-place
 * form).  Supported D as for dan_ln_modulate.  Returns DAN_EINVAL for a bad
 * qscale, otherwise as dan_ln_modulate. */
int dan_ln_modulate_fp8(const dan_bf16 *x, const dan_bf16 *scale, const dan_bf16 *shift,
                        int64_t vec_bstride, float qscale, uint8_t *q, int64_t B, int64_t T,
                        int64_t D, float eps, void *stream);
int dan_can_use_ln_modulate_fp8(const dan_bf16 *x, const dan_bf16 *scale, const dan_bf16 *shift,
                                int64_t vec_bstride, float qscale, const uint8_t *q, int64_t B,
                                int64_t T, int64_t D, float eps);

/* ------------------------------------------- QK-RMSNorm + RoPE epilogue
 * Two token streams (text, then image), each given as three row-strided
 * views q, k, v of [T_s, heads*hd] bf16 (hd = head_dim, 128 or 64) that
 * share one row stride (`*_row_stride` elements, >= heads*hd, a multiple of
 * 8; e.g. the column slices of a packed [T_s, 3*heads*hd] QKV GEMM output,
 * or separate contiguous tensors).  Heads are contiguous hd-element blocks.
 * For every token t and head h of Q and of K:
 *   rstd = rn(1/rn(sqrt(rn(rn(s/hd) + eps_stream)))), s folded from hd/8
 *          logical threads (thread l sums columns 8l..8l+7 in order) by the
 *          adjacent-pair tree,
 *   n_j  = bf16(rn(rn(x_j * rstd) * w_j))   (w: that stream's q or k weight [hd])
 *   out_{2i}   = bf16(rn(rn(n_{2i} * c_i) - rn(n_{2i+1} * s_i)))
 *   out_{2i+1} = bf16(rn(rn(n_{2i} * s_i) + rn(n_{2i+1} * c_i)))
 * (interleaved pairs, the Qwen epilogue's is_neox=False) with c_i =
 * rope[t][i], s_i = rope[t][hd/2 + i] (fp32 rows [cos_0..cos_{hd/2-1} |
 * sin_0..] of that stream's table, row stride hd).  V heads are copied
 * unchanged.  Outputs q_out, k_out, v_out are contiguous
 * [T_txt + T_img, heads, hd], text tokens first.  head_dim 128 or 64
 * (DAN_EUNSUPPORTED otherwise); heads >= 1; T_txt, T_img >= 0; a stream
 * with T_s == 0 may pass NULL pointers for its inputs. */
int dan_qk_norm_rope_epilogue(const dan_bf16 *q_txt, const dan_bf16 *k_txt, const dan_bf16 *v_txt,
                              int64_t T_txt, int64_t txt_row_stride, const dan_bf16 *q_img,
                              const dan_bf16 *k_img, const dan_bf16 *v_img, int64_t T_img,
                              int64_t img_row_stride, int64_t heads, int64_t head_dim,
                              const dan_bf16 *wq_txt, const dan_bf16 *wk_txt,
                              const dan_bf16 *wq_img, const dan_bf16 *wk_img,
                              const float *rope_txt, const float *rope_img, float eps_txt,
                              float eps_img, dan_bf16 *q_out, dan_bf16 *k_out, dan_bf16 *v_out,
                              void *stream);
int dan_can_use_qk_norm_rope_epilogue(
    const dan_bf16 *q_txt, const dan_bf16 *k_txt, const dan_bf16 *v_txt, int64_t T_txt,
    int64_t txt_row_stride, const dan_bf16 *q_img, const dan_bf16 *k_img, const dan_bf16 *v_img,
    int64_t T_img, int64_t img_row_stride, int64_t heads, int64_t head_dim,
    const dan_bf16 *wq_txt, const dan_bf16 *wk_txt, const dan_bf16 *wq_img,
    const dan_bf16 *wk_img, const float *rope_txt, const float *rope_img, float eps_txt,
    float eps_img, const dan_bf16 *q_out, const dan_bf16 *k_out, const dan_bf16 *v_out);

/* The same epilogue with the neox rotation of halves ("rotate half"): for
 * i < hd/2 the pair is (i, i + hd/2),
 *   out_i        = bf16(rn(rn(n_i * c_i) - rn(n_{i+hd/2} * s_i)))
 *   out_{i+hd/2} = bf16(rn(rn(n_i * s_i) + rn(n_{i+hd/2} * c_i)))
 * with the same table rows; everything else as dan_qk_norm_rope_epilogue.
 * The guide lists QK-norm + RoPE variants for other DiTs (FLUX.2, ERNIE);
 * this is the rotation they use when is_neox is set. */
int dan_qk_norm_rope_neox_epilogue(const dan_bf16 *q_txt, const dan_bf16 *k_txt,
                                   const dan_bf16 *v_txt, int64_t T_txt, int64_t txt_row_stride,
                                   const dan_bf16 *q_img, const dan_bf16 *k_img,
                                   const dan_bf16 *v_img, int64_t T_img, int64_t img_row_stride,
                                   int64_t heads, int64_t head_dim, const dan_bf16 *wq_txt,
                                   const dan_bf16 *wk_txt, const dan_bf16 *wq_img,
                                   const dan_bf16 *wk_img, const float *rope_txt,
                                   const float *rope_img, float eps_txt, float eps_img,
                                   dan_bf16 *q_out, dan_bf16 *k_out, dan_bf16 *v_out, void *stream);
int dan_can_use_qk_norm_rope_neox_epilogue(
    const dan_bf16 *q_txt, const dan_bf16 *k_txt, const dan_bf16 *v_txt, int64_t T_txt,
    int64_t txt_row_stride, const dan_bf16 *q_img, const dan_bf16 *k_img, const dan_bf16 *v_img,
    int64_t T_img, int64_t img_row_stride, int64_t heads, int64_t head_dim,
    const dan_bf16 *wq_txt, const dan_bf16 *wk_txt, const dan_bf16 *wq_img,
    const dan_bf16 *wk_img, const float *rope_txt, const float *rope_img, float eps_txt,
    float eps_img, const dan_bf16 *q_out, const dan_bf16 *k_out, const dan_bf16 *v_out);

#ifdef __cplusplus
}
#endif

#endif /* DAN_H */
