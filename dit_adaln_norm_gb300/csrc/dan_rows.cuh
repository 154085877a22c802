// dan_rows.cuh -- fused norm + adaLN modulate row kernels for sm_103a
// (included by dan_rows_rms.cu, dan_rows_gated.cu, dan_rows_ln.cu,
// dan_rows_lnfp8.cu, dan_rows_gatedln.cu and dan_noalloc.cu, which
// instantiate and launch them).
//
// RMSNorm ("SGLang diffusion fused-op package guide", section "Norm +
// scale/shift (adaLN)"; "PR #33854 report", key source excerpt) and
// LayerNorm without affine by Welford ("PR #34126 report", motivation
// section), each followed by the aten modulate chain
// y = bf16(bf16(n * bf16(1 + scale)) + shift).  The gated forms first
// form r' = bf16(r + bf16(gate * h)) and store it; the FP8 form quantises
// y to E4M3 with a static scale.
//
// Design (HBM-bound row work, no tensor cores):
//  - One CTA per SM (two for one shape) takes a contiguous block of rows or
//    every G-th row (G CTAs), whichever measured faster for the shape.  Its
//    warps form teams (one to four warps per row); each team requests its
//    own rows with bulk copies (cp.async.bulk, completion counted on
//    mbarriers, see dan_ring.cuh) into its own shared-memory slots, one or
//    two rows ahead, copies each row from its slot into registers, refills
//    the slot and computes while the next rows are in flight.  Each row is
//    read from HBM once.
//  - Before the dependency wait each team hints its first rows into L2,
//    so that in back-to-back launches they stream while the previous grid
//    drains (the CTA starts as soon as the previous grid's CTA on its SM
//    exits; a prefetch returns nothing to the SM, so it is safe on data the
//    previous grid still writes).
//  - The arithmetic of a row depends only on the row's columns, never on
//    which warp, CTA or launch computes it, so the output bits are
//    independent of B, T and the grid (batch invariance).
//  - bf16(1 + scale), shift, gate and the norm weight are staged in shared
//    memory once per CTA for every batch (when they fit), so the per-element
//    work reads them with conflict-free 16-byte shared loads.  The staging
//    copies are issued before the first rows' loads and completed after
//    them, so the two overlap.
//  - Canonical RMS order: logical thread tx (TPR = D/64 of them) owns the
//    fragments TPR*b + tx (b = 0..7) as one sequential chain; lanes fold by
//    the butterfly (= the adjacent-pair tree); logical warp sums fold by the
//    adjacent-pair tree padded with +0.  A team's warps share the D/2048
//    logical warps of its row.
//  - LayerNorm: 128 logical threads (four logical warps, shared by the
//    team's warps), thread t owns fragments t + 128k; Welford per element with
//    rn(1/n) from a host-computed table; equal-count rows fold in shfl.down
//    order with c = 1/2, ragged rows with the general combine through an
//    ordered xor butterfly; the four warp states fold as (W0 + W2) + (W1 + W3).
#pragma once

#include "dan_device.cuh"
#include "dan_internal.h"
#include "dan_ring.cuh"


namespace dan {

struct RowParams {
    const uint4 *x;
    const uint4 *h;
    const uint4 *scale;
    const uint4 *shift;
    const uint4 *gate;
    const uint4 *weight;
    uint4 *y;
    uint4 *r_out;
    uint2 *q8;   // E4M3 output, 8 codes per 16-byte input fragment (LN + FP8 only)
    float qinv;  // rn(1 / qscale) (LN + FP8 only)
    int64_t rows;
    int64_t T;
    int64_t vs8; // batch stride of the vectors in 16-byte fragments
    int Bs;      // batches staged in shared memory; 0 = read vectors from global
    int F;       // fragments per row (D / 8)
    float eps;
    float inv_d; // 1 / D when D is a power of two (exact), else 0
    unsigned *status;            // device status word (bounded-wait failures)
    unsigned long long limit_ns; // bound of every wait
    unsigned *cta_status;        // per-CTA failure records (CTA_STATUS kernels only)
    int l2_pre;                  // rows per team prefetched into L2 before the dependency wait
    int l2_ahead;                // rows ahead of a slot request prefetched into L2 (0: none)
    int interleave;              // CTA c takes rows c, c + G, ... (else a contiguous block)
    int l2_pre_skip;             // > 1: teams t with t % l2_pre_skip == l2_pre_skip - 1 skip it
};

// Per-batch vector fragment f: which = 0 -> bf16(1 + scale), 1 -> shift,
// 2 -> gate.  Staged copy when available, else computed from global.
template <int NV, bool STAGED>
__device__ __forceinline__ uint4 vec_frag(const RowParams &p, const uint4 *s_vec, int64_t b, int f,
                                          int which)
{
    if (STAGED) return s_vec[(b * NV + which) * p.F + f];
    const int64_t off = b * p.vs8 + f;
    if (which == 0) return one_plus_fragment(ld_vec(p.scale + off));
    return ld_vec((which == 1 ? p.shift : p.gate) + off);
}

// Staging of the norm weight and of scale, shift (, gate) of every batch in
// shared memory, in two halves around the first row loads: stage_begin
// issues asynchronous copies (they enter the memory system ahead of the row
// loads and hold no registers); stage_end waits for them, then rewrites
// each scale fragment in place as bf16(1 + scale).
template <int NV, bool HAS_W>
__device__ __forceinline__ void stage_begin(const RowParams &p, uint4 *s_w, uint4 *s_vec)
{
    const int F = p.F;
    if (HAS_W)
        for (int f = threadIdx.x; f < F; f += blockDim.x) cp_async16(s_w + f, p.weight + f);
    for (int i = threadIdx.x; i < p.Bs * F; i += blockDim.x) {
        const int b = i / F, f = i - b * F;
        const int64_t off = (int64_t)b * p.vs8 + f;
        uint4 *dst = s_vec + (int64_t)b * NV * F;
        cp_async16(dst + f, p.scale + off);
        cp_async16(dst + F + f, p.shift + off);
        if (NV == 3) cp_async16(dst + 2 * F + f, p.gate + off);
    }
    cp_async_commit();
}

template <int NV>
__device__ __forceinline__ void stage_end(const RowParams &p, uint4 *s_vec)
{
    const int F = p.F;
    cp_async_wait_all();
    __syncthreads();
    for (int i = threadIdx.x; i < p.Bs * F; i += blockDim.x) {
        const int b = i / F, f = i - b * F;
        uint4 *dst = s_vec + (int64_t)b * NV * F + f;
        *dst = one_plus_fragment(*dst);
    }
    __syncthreads();
}

// Normalise + modulate one fragment of x with the row's rstd and store it.
template <bool HAS_W>
__device__ __forceinline__ uint4 rms_out_fragment(const uint4 &xv, float rstd, const uint4 &o,
                                                  const uint4 &sh, const uint4 &wv)
{
    uint4 out;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const uint32_t xw = word(xv, i);
        float t0 = __fmul_rn(lo_f(xw), rstd), t1 = __fmul_rn(hi_f(xw), rstd);
        if (HAS_W) {
            const uint32_t ww = word(wv, i);
            t0 = __fmul_rn(t0, lo_f(ww));
            t1 = __fmul_rn(t1, hi_f(ww));
        }
        set_word(out, i, modulate_word(pack_bf16(t0, t1), word(o, i), word(sh, i)));
    }
    return out;
}

// ------------------------------------------------------------------ RMS

// Fragment index of logical thread (chain j, lane), fragment b, RMS order.
template <int LW>
__device__ __forceinline__ int rms_frag(int j, int b, int lane)
{
    return (32 * LW) * b + 32 * j + lane;
}

// The eight bf16 elements of a fragment widened to fp32 (exact).  A row's
// part is widened once, when it is copied out of its slot, and both the
// statistics and the normalisation read the fp32 values.
__device__ __forceinline__ void widen8(const uint4 &f, float (&o)[8])
{
#pragma unroll
    for (int w = 0; w < 4; ++w) {
        o[2 * w] = lo_f(word(f, w));
        o[2 * w + 1] = hi_f(word(f, w));
    }
}

// Packed operations take one element from each of two logical warps (j, j+1)
// when a lane holds an even number of them, else two neighbouring elements
// of one logical warp; the statistics and the normalisation pair them the
// same way, so each pair stays in one register pair.

// Canonical sum of squares of LWW logical warps of a row held in x: one
// ordered chain per logical thread (v fastest, then the fragment index),
// then the butterfly over the 32 lanes (= the adjacent-pair tree).  Every
// lane ends with each logical warp's sum.
template <int LWW>
__device__ __forceinline__ void rms_sums(const float (&x)[LWW][8][8], float (&acc)[LWW])
{
    static_assert(LWW == 1 || LWW % 2 == 0, "one or an even number of logical warps");
    if (LWW == 1) {
        float a = 0.0f;
#pragma unroll
        for (int k = 0; k < 8; ++k)
#pragma unroll
            for (int e = 0; e < 8; e += 2) {
                const float2 x2 = make_float2(x[0][k][e], x[0][k][e + 1]);
                const float2 p = mul2(x2, x2); // two products of one chain, added in order
                a = __fadd_rn(a, p.x);
                a = __fadd_rn(a, p.y);
            }
        acc[0] = a;
    } else {
        constexpr int NP = LWW / 2;
        float2 acc2[NP > 0 ? NP : 1];
#pragma unroll
        for (int q = 0; q < NP; ++q) acc2[q] = make_float2(0.0f, 0.0f);
#pragma unroll
        for (int k = 0; k < 8; ++k)
#pragma unroll
            for (int e = 0; e < 8; ++e)
#pragma unroll
                for (int q = 0; q < NP; ++q) {
                    const float2 x2 = make_float2(x[2 * q][k][e], x[2 * q + 1][k][e]);
                    acc2[q] = addmul2(acc2[q], x2, x2);
                }
#pragma unroll
        for (int q = 0; q < NP; ++q) {
            acc[2 * q] = acc2[q].x;
            acc[2 * q + 1] = acc2[q].y;
        }
    }
#pragma unroll
    for (int off = 1; off < 32; off <<= 1)
#pragma unroll
        for (int j = 0; j < LWW; ++j) acc[j] = __fadd_rn(acc[j], __shfl_xor_sync(kFull, acc[j], off));
}

// rstd of a row from its LW logical warp sums: the adjacent-pair tree padded
// with +0, then rn(1 / rn(sqrt(rn(rn(s / D) + eps)))).
template <int LW>
__device__ __forceinline__ float rms_rstd(const float (&sums)[LW], float eps)
{
    constexpr int P2 = LW <= 1 ? 1 : LW <= 2 ? 2 : 4;
    constexpr int D = 2048 * LW;
    float t[P2];
#pragma unroll
    for (int k = 0; k < P2; ++k) t[k] = k < LW ? sums[k] : 0.0f;
#pragma unroll
    for (int off = 1; off < P2; off <<= 1)
#pragma unroll
        for (int k = 0; k < P2; k += 2 * off) t[k] = __fadd_rn(t[k], t[k + off]);
    return defined_rsqrt(__fadd_rn(div_by<D>(t[0]), eps));
}

// Modulate two rows of normalised fp32 values t[e] (one fragment) and store:
// y = bf16(bf16(bf16(t) * o) + shift).
__device__ __forceinline__ void modulate_store(uint4 *dst, const float (&t)[8], const uint4 &o,
                                               const uint4 &sh)
{
    uint4 out;
#pragma unroll
    for (int w = 0; w < 4; ++w)
        set_word(out, w, modulate_word(pack_bf16(t[2 * w], t[2 * w + 1]), word(o, w), word(sh, w)));
    st_stream(dst, out);
}

// The same modulate, then the static FP8 quantisation of each bf16 result:
// q = e4m3(rn(y * qinv)), nearest even, saturated to +-448; eight codes (8 B)
// per fragment.
__device__ __forceinline__ void modulate_store_fp8(uint2 *dst, const float (&t)[8], const uint4 &o,
                                                   const uint4 &sh, float2 qinv2)
{
    uint32_t codes[4];
#pragma unroll
    for (int w = 0; w < 4; ++w) {
        const uint32_t y = modulate_word(pack_bf16(t[2 * w], t[2 * w + 1]), word(o, w), word(sh, w));
        codes[w] = fp8x2_e4m3(mul2(wide2(y), qinv2));
    }
    st_stream8(dst, make_uint2(codes[0] | (codes[1] << 16), codes[2] | (codes[3] << 16)));
}

// Normalise, modulate and store the logical warps j0 .. j0+LWW-1 of a row
// (for the gated form x already holds r').
template <int LW, int LWW, int NV, bool HAS_W, bool STAGED>
__device__ __forceinline__ void rms_store(const float (&x)[LWW][8][8], int j0, float rstd,
                                          const RowParams &p, int64_t row, int64_t bidx,
                                          const uint4 *s_w, const uint4 *s_vec, int lane)
{
    constexpr int F = 8 * 32 * LW;
    const float2 rstd2 = dup2(rstd);
    uint4 *y = p.y + row * F;
    if (LWW == 1) {
#pragma unroll
        for (int k = 0; k < 8; ++k) {
            const int f = rms_frag<LW>(j0, k, lane);
            uint4 wv = make_uint4(0, 0, 0, 0);
            if (HAS_W) wv = s_w[f];
            float t[8];
#pragma unroll
            for (int e = 0; e < 8; e += 2) {
                float2 t2 = mul2(make_float2(x[0][k][e], x[0][k][e + 1]), rstd2);
                if (HAS_W) t2 = mul2(t2, wide2(word(wv, e / 2)));
                t[e] = t2.x;
                t[e + 1] = t2.y;
            }
            modulate_store(y + f, t, vec_frag<NV, STAGED>(p, s_vec, bidx, f, 0),
                           vec_frag<NV, STAGED>(p, s_vec, bidx, f, 1));
        }
    } else {
#pragma unroll
        for (int q = 0; q < LWW / 2; ++q)
#pragma unroll
            for (int k = 0; k < 8; ++k) {
                const int f0 = rms_frag<LW>(j0 + 2 * q, k, lane);
                const int f1 = rms_frag<LW>(j0 + 2 * q + 1, k, lane);
                uint4 w0 = make_uint4(0, 0, 0, 0), w1 = w0;
                if (HAS_W) {
                    w0 = s_w[f0];
                    w1 = s_w[f1];
                }
                float t0[8], t1[8];
#pragma unroll
                for (int e = 0; e < 8; ++e) {
                    float2 t2 = mul2(make_float2(x[2 * q][k][e], x[2 * q + 1][k][e]), rstd2);
                    if (HAS_W) t2 = mul2(t2, make_float2(elem(w0, e), elem(w1, e)));
                    t0[e] = t2.x;
                    t1[e] = t2.y;
                }
                modulate_store(y + f0, t0, vec_frag<NV, STAGED>(p, s_vec, bidx, f0, 0),
                               vec_frag<NV, STAGED>(p, s_vec, bidx, f0, 1));
                modulate_store(y + f1, t1, vec_frag<NV, STAGED>(p, s_vec, bidx, f1, 0),
                               vec_frag<NV, STAGED>(p, s_vec, bidx, f1, 1));
            }
    }
}

// ------------------------------------------------------------ LayerNorm

struct Welford {
    float n, mean, m2;
};

// Count-weighted combine of A (lower lane / warp) and B; empty sides pass.
__device__ __forceinline__ Welford combine(const Welford &A, const Welford &B)
{
    if (B.n == 0.0f) return A;
    if (A.n == 0.0f) return B;
    Welford o;
    o.n = __fadd_rn(A.n, B.n);
    const float c = (A.n == B.n) ? 0.5f : __fdiv_rn(B.n, o.n); // rn(nB/n); exact 1/2 if equal
    const float delta = __fsub_rn(B.mean, A.mean);
    o.mean = __fadd_rn(A.mean, __fmul_rn(delta, c));
    o.m2 = __fadd_rn(__fadd_rn(A.m2, B.m2), __fmul_rn(__fmul_rn(__fmul_rn(delta, delta), A.n), c));
    return o;
}

// The same combine for two states of equal count nA (so c = nB/n = 1/2
// exactly), on packed pairs of independent states.
__device__ __forceinline__ void combine_eq2(float2 &meanA, float2 &m2A, const float2 &meanB,
                                            const float2 &m2B, float nA)
{
    const float2 half = dup2(0.5f);
    const float2 delta = sub2(meanB, meanA);
    meanA = addmul2(meanA, delta, half);
    m2A = addmul2(add2(m2A, m2B), mul2(mul2(delta, delta), dup2(nA)), half);
}

__device__ __forceinline__ void combine_eq1(float &meanA, float &m2A, float meanB, float m2B,
                                            float nA)
{
    const float delta = __fsub_rn(meanB, meanA);
    meanA = __fadd_rn(meanA, __fmul_rn(delta, 0.5f));
    m2A = __fadd_rn(__fadd_rn(m2A, m2B), __fmul_rn(__fmul_rn(__fmul_rn(delta, delta), nA), 0.5f));
}

// Fold the 32 lanes of a logical warp in shfl.down order; every lane ends
// with lane 0's result (each pair computes the same ordered combine).
__device__ __forceinline__ Welford warp_fold(Welford s, int lane)
{
#pragma unroll
    for (int off = 16; off >= 1; off >>= 1) {
        Welford o;
        o.n = __shfl_xor_sync(kFull, s.n, off);
        o.mean = __shfl_xor_sync(kFull, s.mean, off);
        o.m2 = __shfl_xor_sync(kFull, s.m2, off);
        const bool lower = (lane & off) == 0;
        s = lower ? combine(s, o) : combine(o, s);
    }
    return s;
}

// rn(1/n) for n = 1..64 as duplicated pairs (host IEEE division).
struct InvTable2 {
    float2 v[65];
};

// Fragment of logical thread t = 32j + lane at its k-th visit: t + 128k.
__device__ __forceinline__ int ln_frag(int j, int lane, int k) { return 32 * j + lane + 128 * k; }

// Welford states of the J logical warps j = r + TW*m (m = 0..J-1) of a row
// held in x, each folded over its 32 threads in the canonical order; every
// lane ends with the states.
template <int FPT, int J, int TW, bool RAGGED>
__device__ __forceinline__ void ln_states(const float (&x)[J][FPT][8], int r, int F,
                                          const InvTable2 &inv, int lane, Welford (&W)[J])
{
    if (!RAGGED) {
        // Every logical thread holds FPT full fragments: counts are equal
        // everywhere, so each combine has c = 1/2 exactly.  Logical warps
        // m, m+1 of a lane share packed operations.
        constexpr int NP = J / 2;
        float2 mean2[NP > 0 ? NP : 1], m22[NP > 0 ? NP : 1];
        float mean1 = 0.0f, m21 = 0.0f;
#pragma unroll
        for (int q = 0; q < NP; ++q) mean2[q] = m22[q] = make_float2(0.0f, 0.0f);
        // rn(1/n) from the host table, or for two-warp teams at D <= 4096 as
        // the compile-time constant 1.0f / n (the same IEEE quotient; it
        // measured faster there, 8.06 against 8.25 us for the CFG batch
        // [2,1140,4096], and slower with single-warp teams, 9.38 against 9.22
        // at [1,4096,3072])
        constexpr bool kImmRcp = TW == 2 && FPT <= 4;
#pragma unroll
        for (int k = 0; k < FPT; ++k)
#pragma unroll
            for (int e = 0; e < 8; ++e) {
                const float2 rr = kImmRcp ? dup2(1.0f / (float)(8 * k + e + 1)) : inv.v[8 * k + e + 1];
#pragma unroll
                for (int q = 0; q < NP; ++q) {
                    const float2 x2 = make_float2(x[2 * q][k][e], x[2 * q + 1][k][e]);
                    const float2 d = sub2(x2, mean2[q]);
                    mean2[q] = addmul2(mean2[q], d, rr);
                    m22[q] = addmul2(m22[q], d, sub2(x2, mean2[q]));
                }
                if (J & 1) {
                    const float xv = x[J - 1][k][e];
                    const float d = __fsub_rn(xv, mean1);
                    mean1 = __fadd_rn(mean1, __fmul_rn(d, rr.x));
                    m21 = __fadd_rn(m21, __fmul_rn(d, __fsub_rn(xv, mean1)));
                }
            }
        float nA = (float)(8 * FPT);
#pragma unroll
        for (int off = 16; off >= 1; off >>= 1) {
#pragma unroll
            for (int q = 0; q < NP; ++q) {
                const float2 mb = make_float2(__shfl_down_sync(kFull, mean2[q].x, off),
                                              __shfl_down_sync(kFull, mean2[q].y, off));
                const float2 m2b = make_float2(__shfl_down_sync(kFull, m22[q].x, off),
                                               __shfl_down_sync(kFull, m22[q].y, off));
                combine_eq2(mean2[q], m22[q], mb, m2b, nA);
            }
            if (J & 1) {
                const float mb = __shfl_down_sync(kFull, mean1, off);
                const float m2b = __shfl_down_sync(kFull, m21, off);
                combine_eq1(mean1, m21, mb, m2b, nA);
            }
            nA = 2.0f * nA;
        }
        const float nw = (float)(256 * FPT);
#pragma unroll
        for (int q = 0; q < NP; ++q) {
            W[2 * q] = Welford{nw, __shfl_sync(kFull, mean2[q].x, 0), __shfl_sync(kFull, m22[q].x, 0)};
            W[2 * q + 1] =
                Welford{nw, __shfl_sync(kFull, mean2[q].y, 0), __shfl_sync(kFull, m22[q].y, 0)};
        }
        if (J & 1) W[J - 1] = Welford{nw, __shfl_sync(kFull, mean1, 0), __shfl_sync(kFull, m21, 0)};
    } else {
#pragma unroll
        for (int m = 0; m < J; ++m) {
            const int j = r + TW * m;
            float mean = 0.0f, m2 = 0.0f;
            int nfr = 0;
#pragma unroll
            for (int k = 0; k < FPT; ++k) {
                if (ln_frag(j, lane, k) < F) {
                    nfr = k + 1;
#pragma unroll
                    for (int e = 0; e < 8; ++e) {
                        const float xv = x[m][k][e];
                        const float d = __fsub_rn(xv, mean);
                        mean = __fadd_rn(mean, __fmul_rn(d, inv.v[8 * k + e + 1].x));
                        m2 = __fadd_rn(m2, __fmul_rn(d, __fsub_rn(xv, mean)));
                    }
                }
            }
            W[m] = warp_fold(Welford{(float)(8 * nfr), mean, m2}, lane);
        }
    }
}

// Mean and m2 of a row from its four logical warp states: (W0 + W2) + (W1 + W3).
template <bool RAGGED>
__device__ __forceinline__ void ln_final(const Welford (&W)[4], float &mean, float &m2)
{
    if (!RAGGED) {
        const float nw = W[0].n; // all four counts are equal
        float2 m01 = make_float2(W[0].mean, W[1].mean), q01 = make_float2(W[0].m2, W[1].m2);
        combine_eq2(m01, q01, make_float2(W[2].mean, W[3].mean), make_float2(W[2].m2, W[3].m2), nw);
        mean = m01.x;
        m2 = q01.x;
        combine_eq1(mean, m2, m01.y, q01.y, 2.0f * nw);
    } else {
        const Welford S = combine(combine(W[0], W[2]), combine(W[1], W[3]));
        mean = S.mean;
        m2 = S.m2;
    }
}

// Normalise, modulate and store (FP8: quantise and store) the logical warps
// r + TW*m of a row.
template <int FPT, int J, int TW, bool RAGGED, bool STAGED, bool FP8, int NV>
__device__ __forceinline__ void ln_store(const float (&x)[J][FPT][8], int r, float mean, float m2,
                                         const RowParams &p, int64_t row, int64_t bidx,
                                         const uint4 *s_vec, int lane)
{
    const int F = p.F;
    // rn(m2 / D): a multiply by the exact reciprocal when D is a power of
    // two (the same bits as the division), else the IEEE division
    const float var = p.inv_d != 0.0f ? __fmul_rn(m2, p.inv_d) : __fdiv_rn(m2, (float)(8 * F));
    const float2 rstd2 = dup2(defined_rsqrt(__fadd_rn(var, p.eps)));
    const float2 mean2 = dup2(mean);
    uint4 *y = FP8 ? nullptr : p.y + row * F;
    uint2 *q8 = FP8 ? p.q8 + row * F : nullptr;
    const float2 qinv2 = dup2(p.qinv);
    auto out = [&](int f, const float (&t)[8]) {
        const uint4 o = vec_frag<NV, STAGED>(p, s_vec, bidx, f, 0);
        const uint4 sh = vec_frag<NV, STAGED>(p, s_vec, bidx, f, 1);
        if (FP8) modulate_store_fp8(q8 + f, t, o, sh, qinv2);
        else modulate_store(y + f, t, o, sh);
    };
    if (!RAGGED && J >= 2) { // pairs across logical warps, as in ln_states
#pragma unroll
        for (int q = 0; q < J / 2; ++q)
#pragma unroll
            for (int k = 0; k < FPT; ++k) {
                const int f0 = ln_frag(r + TW * 2 * q, lane, k);
                const int f1 = ln_frag(r + TW * (2 * q + 1), lane, k);
                float t0[8], t1[8];
#pragma unroll
                for (int e = 0; e < 8; ++e) {
                    const float2 t2 =
                        mul2(sub2(make_float2(x[2 * q][k][e], x[2 * q + 1][k][e]), mean2), rstd2);
                    t0[e] = t2.x;
                    t1[e] = t2.y;
                }
                out(f0, t0);
                out(f1, t1);
            }
    } else { // neighbouring elements of one logical warp
#pragma unroll
        for (int m = 0; m < J; ++m)
#pragma unroll
            for (int k = 0; k < FPT; ++k) {
                const int f = ln_frag(r + TW * m, lane, k);
                if (RAGGED && f >= F) continue;
                float t[8];
#pragma unroll
                for (int e = 0; e < 8; e += 2) {
                    const float2 t2 = mul2(sub2(make_float2(x[m][k][e], x[m][k][e + 1]), mean2), rstd2);
                    t[e] = t2.x;
                    t[e + 1] = t2.y;
                }
                out(f, t);
            }
    }
}

// ------------------------------------------------------- the row kernel

enum RowKind { kRms = 0, kGated = 1, kLn = 2, kLnFp8 = 3, kGatedLn = 4 };

template <int KIND>
struct RowShape {
    static constexpr bool GATED = KIND == kGated || KIND == kGatedLn;
    static constexpr int NIN = GATED ? 2 : 1; // bulk-copied inputs per row
    static constexpr int NV = GATED ? 3 : 2;  // staged vectors per batch
};

// Team exchange: per team and row parity, the logical warp results of a
// row (RMS: LW sums; LayerNorm: four states of n, mean, m2).
constexpr int kXchFloats = 16;

// Shared memory: NT = NW / TW teams of TW warps; each team owns SPC row
// slots (NIN inputs of D bf16 each); then the norm weight, the staged
// vectors, one mbarrier per slot, two team mbarriers per team (slot read,
// results published), and the team exchange area.
template <int KIND, int NW, int TW, int SPC>
struct RowLayout {
    static constexpr int NT = NW / TW;
    static int64_t slots_bytes(int F) { return (int64_t)NT * SPC * RowShape<KIND>::NIN * F * 16; }
    static constexpr int tail_bytes = NT * SPC * 8 + 2 * NT * 8 + NT * 2 * kXchFloats * 4;
};

// CTA c takes the contiguous rows [c*R/G, (c+1)*R/G), or with p.interleave
// the rows c, c + G, c + 2G, ...  Its warps form NT = NW / TW teams; team t
// takes the CTA's rows t, t + NT, t + 2NT, ... (in that order of the CTA's
// rows) one at a time and requests each row SPC rows ahead into its own slots
// (dan_ring.cuh).  A row's logical warps (LW for RMS, 4 for LayerNorm) are
// shared among the team's warps, each holding its part in registers.  The
// leader refills a slot once every warp of the team has read it (team
// mbarrier `read`); the warps exchange their logical warp sums or states
// through shared memory (team mbarrier `done`), and each combines all of
// them in the canonical order, so the result does not depend on TW.  Every
// wait is bounded.
// CTA_STATUS kernels also keep one failure record per CTA in
// p.cta_status[blockIdx.x], cleared when the CTA starts.  CPS CTAs share an
// SM (the register budget is set for that many).
template <int KIND, int LW, int FPT, int NW, int TW, int SPC, bool HAS_W, bool RAGGED,
          bool STAGED, bool CTA_STATUS = false, int CPS = 1>
__global__ void __launch_bounds__(32 * NW, CPS)
    row_ring_kernel(const RowParams p, const InvTable2 inv)
{
    using Shape = RowShape<KIND>;
    using Pipe = WarpPipe<SPC>;
    using Lay = RowLayout<KIND, NW, TW, SPC>;
    constexpr int NIN = Shape::NIN, NV = Shape::NV, NT = Lay::NT;
    constexpr bool LN = KIND == kLn || KIND == kLnFp8 || KIND == kGatedLn;
    constexpr int LWW = LN ? 1 : LW / TW; // RMS logical warps per warp
    constexpr int J = LN ? 4 / TW : 1;     // LayerNorm logical warps per warp
    static_assert(NW % TW == 0, "teams of TW warps");
    static_assert(LN ? (4 % TW == 0) : (LW % TW == 0), "TW divides the logical warps");
    const int F = p.F;
    const unsigned row_bytes = (unsigned)F * 16u;

    extern __shared__ __align__(128) uint4 smem[];
    uint4 *ring = smem;                                // NT * SPC * NIN * F
    uint4 *s_w = ring + (int64_t)NT * SPC * NIN * F;   // F if HAS_W
    uint4 *s_vec = s_w + (HAS_W ? F : 0);              // Bs * NV * F
    uint64_t *full = reinterpret_cast<uint64_t *>(s_vec + (int64_t)p.Bs * NV * F);
    uint64_t *read_bar = full + NT * SPC; // per team: every warp has read the slot
    uint64_t *done_bar = read_bar + NT;    // per team: every warp has published its results
    float *xch_all = reinterpret_cast<float *>(done_bar + NT);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int team = warp / TW, r = warp % TW;
    const int64_t G = gridDim.x;
    // the team's rows: rbase + rstep * i for i < units
    int64_t rbase, rstep, rend;
    if (p.interleave) {
        rbase = blockIdx.x + G * team;
        rstep = G * NT;
        rend = p.rows;
    } else {
        const int64_t r0 = (int64_t)blockIdx.x * p.rows / G;
        rbase = r0 + team;
        rstep = NT;
        rend = (int64_t)(blockIdx.x + 1) * p.rows / G;
    }
    const int units = rbase < rend ? (int)((rend - rbase + rstep - 1) / rstep) : 0;
    const bool leader = r == 0 && lane == 0;
    // L2 prefetch of the team's row i: its first l2_pre rows before the
    // dependency wait, so that they stream while the previous grid drains;
    // with l2_ahead > 0 also row i + SPC + l2_ahead when row i + SPC is
    // requested into its slot.
    auto prefetch = [&](int i) { // the team leader only
        const int64_t row = rbase + rstep * i;
        prefetch_l2(p.x + row * F, row_bytes);
        if (NIN == 2) prefetch_l2(p.h + row * F, row_bytes);
    };
    if (leader)
        for (int i = 0; i < p.l2_pre && i < units; ++i) {
            if (p.l2_pre_skip > 1 && team % p.l2_pre_skip == p.l2_pre_skip - 1) break;
            prefetch(i);
        }
    if (threadIdx.x == 32 && p.Bs > 0) { // the staged vectors, likewise
        if (HAS_W) prefetch_l2(p.weight, row_bytes);
        for (int b = 0; b < p.Bs; ++b) {
            prefetch_l2(p.scale + (int64_t)b * p.vs8, row_bytes);
            prefetch_l2(p.shift + (int64_t)b * p.vs8, row_bytes);
            if (NV == 3) prefetch_l2(p.gate + (int64_t)b * p.vs8, row_bytes);
        }
    }

    if (threadIdx.x == 0) {
        for (int s = 0; s < NT * SPC; ++s) mbar_init(full + s, 1);
        for (int t = 0; t < NT; ++t) {
            mbar_init(read_bar + t, TW);
            mbar_init(done_bar + t, TW);
        }
        mbar_init_fence();
    }
    grid_dependency_wait(); // no global read above this line (L2 prefetches only)
    allow_dependents();
    if (CTA_STATUS && threadIdx.x == 0) p.cta_status[blockIdx.x] = 0u;
    stage_begin<NV, HAS_W>(p, s_w, s_vec);
    __syncthreads(); // barriers initialised

    uint4 *slots = ring + (int64_t)team * SPC * NIN * F;
    uint64_t *bar = full + team * SPC;
    auto request = [&](int i) { // the team leader only
        const int64_t row = rbase + rstep * i;
        uint4 *dst = slots + (int64_t)Pipe::slot(i) * NIN * F;
        uint64_t *b = bar + Pipe::slot(i);
        mbar_arrive_expect_tx(b, NIN * row_bytes);
        bulk_load(dst, p.x + row * F, row_bytes, b);
        if (NIN == 2) bulk_load(dst + F, p.h + row * F, row_bytes, b);
    };
    auto fail = [&](int i) {
        const unsigned bits = Pipe::abort(bar, i, units, p.status, p.limit_ns);
        if (CTA_STATUS) set_status(p.cta_status + blockIdx.x, bits);
    };
    // The first SPC rows go out before waiting for the staged vectors.
    if (leader)
        for (int i = 0; i < SPC && i < units; ++i) request(i);
    stage_end<NV>(p, s_vec);

    // Batch of the team's current row, kept incrementally (rows step by
    // rstep = q_step * T + r_step).
    int64_t bidx = 0, t_in = 0, q_step = 0, r_step = 0;
    if (units > 0) {
        bidx = rbase / p.T;
        t_in = rbase - bidx * p.T;
        q_step = rstep / p.T;
        r_step = rstep - q_step * p.T;
    }
    for (int i = 0; i < units; ++i) {
        if (i > 0) {
            bidx += q_step;
            t_in += r_step;
            if (t_in >= p.T) {
                t_in -= p.T;
                ++bidx;
            }
        }
        if (!Pipe::wait(bar, i, p.limit_ns)) {
            fail(i);
            return;
        }
        const uint4 *src = slots + (int64_t)Pipe::slot(i) * NIN * F;
        const int64_t row = rbase + rstep * i;
        float *xch = xch_all + (team * 2 + (i & 1)) * kXchFloats;
        // After this warp has read the slot (slot_reads_done): the leader
        // refills it once every warp of the team has read it.  A warp
        // arrives on `read` for row i+1 only after `done` of row i, which
        // needs the leader's arrivals of row i, so the phases never mix.
        auto refill = [&]() -> bool {
            if (TW > 1) {
                if (lane == 0) mbar_arrive(read_bar + team);
                if (r == 0 && !mbar_wait(read_bar + team, (unsigned)i & 1u, p.limit_ns))
                    return false;
            }
            if (leader && i + SPC < units) {
                request(i + SPC);
                if (p.l2_ahead > 0 && i + SPC + p.l2_ahead < units) prefetch(i + SPC + p.l2_ahead);
            }
            return true;
        };
        // Teams of several warps: publish this warp's results (written to
        // xch by lane 0) and wait for the other warps'.
        auto publish = [&]() -> bool {
            if (TW == 1) return true;
            __syncwarp();
            if (lane == 0) mbar_arrive(done_bar + team);
            return mbar_wait(done_bar + team, (unsigned)i & 1u, p.limit_ns);
        };
        if (LN) {
            float x[J][FPT][8];
#pragma unroll
            for (int m = 0; m < J; ++m)
#pragma unroll
                for (int q = 0; q < FPT; ++q) {
                    const int f = ln_frag(r + TW * m, lane, q);
                    uint4 v = make_uint4(0, 0, 0, 0);
                    if (!RAGGED || f < F) {
                        v = src[f];
                        if (KIND == kGatedLn) { // r' = bf16(r + bf16(gate * h)), stored at once
                            const uint4 g = vec_frag<NV, STAGED>(p, s_vec, bidx, f, 2);
                            const uint4 hh = src[F + f];
                            v = make_uint4(gated_word(v.x, g.x, hh.x), gated_word(v.y, g.y, hh.y),
                                           gated_word(v.z, g.z, hh.z), gated_word(v.w, g.w, hh.w));
                            st_stream(p.r_out + row * F + f, v);
                        }
                    }
                    widen8(v, x[m][q]);
                }
            slot_reads_done();
            if (!refill()) {
                fail(i);
                return;
            }
            Welford W[J];
            ln_states<FPT, J, TW, RAGGED>(x, r, F, inv, lane, W);
            Welford all[4];
            if (TW == 1) {
#pragma unroll
                for (int m = 0; m < 4; ++m) all[m] = W[m % J];
            } else {
                if (lane == 0)
#pragma unroll
                    for (int m = 0; m < J; ++m) {
                        float *o = xch + 3 * (r + TW * m);
                        o[0] = W[m].n;
                        o[1] = W[m].mean;
                        o[2] = W[m].m2;
                    }
            }
            if (!publish()) {
                fail(i);
                return;
            }
            if (TW > 1)
#pragma unroll
                for (int m = 0; m < 4; ++m) all[m] = Welford{xch[3 * m], xch[3 * m + 1], xch[3 * m + 2]};
            float mean, m2;
            ln_final<RAGGED>(all, mean, m2);
            ln_store<FPT, J, TW, RAGGED, STAGED, KIND == kLnFp8, NV>(x, r, mean, m2, p, row, bidx,
                                                                     s_vec, lane);
        } else {
            float x[LWW][8][8];
            const int j0 = r * LWW;
#pragma unroll
            for (int j = 0; j < LWW; ++j)
#pragma unroll
                for (int q = 0; q < 8; ++q) {
                    const int f = rms_frag<LW>(j0 + j, q, lane);
                    uint4 v = src[f];
                    if (KIND == kGated) { // r' = bf16(r + bf16(gate * h)), stored at once
                        const uint4 g = vec_frag<NV, STAGED>(p, s_vec, bidx, f, 2);
                        const uint4 hh = src[F + f];
                        v = make_uint4(gated_word(v.x, g.x, hh.x), gated_word(v.y, g.y, hh.y),
                                       gated_word(v.z, g.z, hh.z), gated_word(v.w, g.w, hh.w));
                        st_stream(p.r_out + row * F + f, v);
                    }
                    widen8(v, x[j][q]);
                }
            slot_reads_done();
            if (!refill()) {
                fail(i);
                return;
            }
            float acc[LWW];
            rms_sums<LWW>(x, acc);
            float sums[LW];
            if (TW == 1) {
#pragma unroll
                for (int j = 0; j < LW; ++j) sums[j] = acc[j % LWW];
            } else if (lane == 0) {
#pragma unroll
                for (int j = 0; j < LWW; ++j) xch[j0 + j] = acc[j];
            }
            if (!publish()) {
                fail(i);
                return;
            }
            if (TW > 1)
#pragma unroll
                for (int j = 0; j < LW; ++j) sums[j] = xch[j];
            rms_store<LW, LWW, NV, HAS_W, STAGED>(x, j0, rms_rstd<LW>(sums, p.eps), p, row, bidx,
                                                  s_w, s_vec, lane);
        }
    }
}

// ------------------------------------------------------------- launching

namespace {

constexpr unsigned long long kWaitLimitNs = 1000000000ull; // 1 s per wait
constexpr int kStageBudget = 96 * 1024; // most shared memory staged vectors may take

// Raise the dynamic shared-memory limit of `fn` the first time it needs more.
template <typename K>
cudaError_t allow_smem(K fn, int smem)
{
    return allow_dynamic_smem(reinterpret_cast<const void *>(fn), smem);
}

RowParams make_params(const RowProblem &q)
{
    RowParams p;
    p.x = static_cast<const uint4 *>(q.x);
    p.h = static_cast<const uint4 *>(q.h);
    p.scale = static_cast<const uint4 *>(q.scale);
    p.shift = static_cast<const uint4 *>(q.shift);
    p.gate = static_cast<const uint4 *>(q.gate);
    p.weight = static_cast<const uint4 *>(q.weight);
    p.y = static_cast<uint4 *>(q.y);
    p.r_out = static_cast<uint4 *>(q.r_out);
    p.q8 = static_cast<uint2 *>(q.q);
    p.qinv = q.qinv;
    p.rows = q.B * q.T;
    p.T = q.T;
    p.vs8 = q.vs / 8;
    p.F = (int)(q.D / 8);
    p.eps = q.eps;
    p.inv_d = (q.D & (q.D - 1)) == 0 ? 1.0f / (float)q.D : 0.0f;
    p.Bs = 0;
    p.status = device_status();
    p.limit_ns = kWaitLimitNs;
    p.cta_status = nullptr;
    p.l2_pre = 0;
    p.l2_ahead = 0;
    p.interleave = 0;
    p.l2_pre_skip = 1;
    return p;
}

InvTable2 inv_table()
{
    InvTable2 inv;
    inv.v[0] = make_float2(0.0f, 0.0f);
    for (int n = 1; n <= 64; ++n) {
        const float r = 1.0f / (float)n; // IEEE division on the host
        inv.v[n] = make_float2(r, r);
    }
    return inv;
}

// Shared memory a launch of row_ring_kernel<KIND, ..., NW, TW, SPC> needs,
// with p.Bs set to the number of batches whose vectors are staged (all of
// them when they fit in the staging budget, else none).  With CPS CTAs per
// SM each CTA keeps to its share of the SM's shared memory.
template <int KIND, int NW, int TW, int SPC, int CPS = 1>
int ring_smem(const RowProblem &q, RowParams &p)
{
    using Shape = RowShape<KIND>;
    using Lay = RowLayout<KIND, NW, TW, SPC>;
    const int64_t row_bytes = q.D * 2;
    const int64_t fixed = Lay::slots_bytes((int)(q.D / 8)) +
                          ((KIND == kRms || KIND == kGated) && q.weight ? row_bytes : 0) +
                          Lay::tail_bytes;
    const int64_t vec_bytes = q.B * Shape::NV * row_bytes;
    const int64_t room = (int64_t)max_smem_optin() / CPS - (CPS > 1 ? 2048 : 0) - fixed;
    p.Bs = (vec_bytes <= kStageBudget && vec_bytes <= room) ? (int)q.B : 0;
    return (int)(fixed + (p.Bs ? vec_bytes : 0));
}

// CTAs of a row launch: CPS per SM (one unless the shape is made for
// several: the slots and the warps' registers fill the SM), at most one per
// row.
inline int ring_grid(int64_t rows, int cps = 1)
{
    const int64_t g = (int64_t)cps * sm_count();
    return (int)(rows < g ? rows : g);
}

// Each CTA takes a contiguous block of rows (or every G-th row with IL).
// Each team prefetches its
// first PRE rows (SPC when PRE is 0) into L2 before the dependency wait,
// and with AHEAD > 0 row i + SPC + AHEAD when it requests row i + SPC.
// CTA_STATUS kernels write one failure record per CTA into `cta_status`,
// which holds `cta_capacity` records: a launch that would need more is
// refused (nothing launched).  CPS CTAs share each SM.  IL: each CTA takes
// every G-th row instead of a contiguous block (G CTAs).  SKIP > 1: every
// SKIP-th team prefetches nothing before the wait, so the first burst is
// smaller and lands sooner and those teams' rows follow it (measured faster
// with SKIP = 3 for every shape measured but RMS at D = 4096: C2' 10.91
// against 11.34 us, C3 20.36 against 20.83, [1,4216,8192] RMS 20.27
// against 20.93; C1' 10.44 against 10.27).
template <int KIND, int LW, int FPT, int NW, int TW, int SPC, bool RAGGED, bool CTA_STATUS = false,
          int PRE = 0, int AHEAD = 0, int CPS = 1, bool IL = false, int SKIP = 3>
cudaError_t launch_ring(const RowProblem &q, cudaStream_t s, unsigned *cta_status = nullptr,
                        int cta_capacity = 0)
{
    RowParams p = make_params(q);
    p.cta_status = cta_status;
    p.l2_pre = PRE > 0 ? PRE : SPC;
    p.l2_ahead = AHEAD;
    p.interleave = IL ? 1 : 0;
    p.l2_pre_skip = SKIP;
    const bool has_w = (KIND == kRms || KIND == kGated) && q.weight != nullptr;
    const int smem = ring_smem<KIND, NW, TW, SPC, CPS>(q, p);
    const int grid = ring_grid(p.rows, CPS);
    if (CTA_STATUS && (cta_status == nullptr || grid > cta_capacity))
        return cudaErrorInvalidConfiguration;
    const InvTable2 inv = inv_table();
    auto go = [&](auto fn) -> cudaError_t {
        const cudaError_t e = allow_smem(fn, smem);
        if (e != cudaSuccess) return e;
        return launch_overlapped(fn, grid, 32 * NW, smem, s, p, inv);
    };
    constexpr bool CS = CTA_STATUS;
    if constexpr (KIND == kRms || KIND == kGated) {
        if (has_w)
            return p.Bs ? go(row_ring_kernel<KIND, LW, FPT, NW, TW, SPC, true, RAGGED, true, CS, CPS>)
                        : go(row_ring_kernel<KIND, LW, FPT, NW, TW, SPC, true, RAGGED, false, CS, CPS>);
    }
    return p.Bs ? go(row_ring_kernel<KIND, LW, FPT, NW, TW, SPC, false, RAGGED, true, CS, CPS>)
                : go(row_ring_kernel<KIND, LW, FPT, NW, TW, SPC, false, RAGGED, false, CS, CPS>);
}

// Problems with at least this many rows per SM use 12 warps per CTA for the
// common widths (three per scheduler: more rows in flight and fewer rows
// per warp); smaller ones do better with 8 (measured).
constexpr int kManyRowsPerSm = 24;
inline bool many_rows(const RowProblem &q)
{
    return q.B * q.T >= (int64_t)kManyRowsPerSm * sm_count();
}

// RMSNorm + modulate shapes (warps NW, warps per row TW, slots per team SPC)
// per width, each CTA taking every G-th row (measured faster than contiguous
// blocks at every width: [1,4216,6144] 15.30 against 15.99 us, 8192 20.70
// against 21.27), chosen by measurement: single-warp teams with two slots each,
// twelve of them when there are many rows per SM and eight otherwise, did
// better than fewer teams with more slots or multi-warp teams at these
// widths; rows of 6144 and 8192 are shared by three and four warps, which
// keeps them in registers.  CTA_STATUS selects the kernels that also write
// per-CTA failure records (see launch_ring).
template <bool CTA_STATUS>
cudaError_t launch_rms_shapes(const RowProblem &q, cudaStream_t s, unsigned *cta_status = nullptr,
                              int cta_capacity = 0)
{
    constexpr bool CS = CTA_STATUS;
    switch (q.D) {
    case 2048:
        return launch_ring<kRms, 1, 8, 8, 1, 2, false, CS, 0, 0, 1, true>(q, s, cta_status, cta_capacity);
    case 4096:
        // one row per team prefetched before the wait (two, one per slot,
        // measured 11.39 against 10.32 us at [1,4216,4096])
        return many_rows(q) ? launch_ring<kRms, 2, 8, 12, 1, 2, false, CS, 1, 0, 1, true, 1>(
                                  q, s, cta_status, cta_capacity)
                            : launch_ring<kRms, 2, 8, 8, 1, 2, false, CS, 0, 0, 1, true, 1>(
                                  q, s, cta_status, cta_capacity);
    case 6144:
        return launch_ring<kRms, 3, 8, 12, 3, 2, false, CS, 0, 0, 1, true>(q, s, cta_status, cta_capacity);
    default: // 8192: 4 warps per row; three rows per team prefetched before the
             // wait, then each row two ahead of the one requested
        return launch_ring<kRms, 4, 8, 16, 4, 1, false, CS, 3, 1, 1, true>(q, s, cta_status, cta_capacity);
    }
}

// LayerNorm shapes (LayerNorm and its FP8 form) by fragments per logical
// thread (D / 1024, rounded up).  At D = 3072 and 4096 with many rows:
// twelve single-warp teams per SM, each CTA taking every G-th row (against
// a contiguous block per CTA: 11.05 against 11.11 us at [1,4216,4096],
// 9.05 against 9.00 and 9.12 against 9.50 us at [1,4096,3072] on two
// GB300s); for the FP8 producer two CTAs of six per SM on contiguous blocks
// (10.82 against 11.10 us at [1,4216,4096], 9.20 against 9.27 at
// [1,4096,3072]; interleaved rows measured 0.1 to 0.25 us slower on one GB300
// and as much faster on another).  With fewer rows: eight two-warp teams.
template <int KIND, int FPT, bool RAGGED>
cudaError_t launch_ln_many(const RowProblem &q, cudaStream_t s)
{
    if constexpr (KIND == kLnFp8) return launch_ring<KIND, 4, FPT, 6, 1, 1, RAGGED, false, 0, 0, 2>(q, s);
    else return launch_ring<KIND, 4, FPT, 12, 1, 1, RAGGED, false, 0, 0, 1, true>(q, s);
}

template <int KIND, bool RAGGED>
cudaError_t launch_ln_fpt(const RowProblem &q, cudaStream_t s)
{
    switch ((q.D + 1023) / 1024) {
    case 1: return launch_ring<KIND, 4, 1, 8, 1, 1, RAGGED>(q, s);
    case 2: return launch_ring<KIND, 4, 2, 8, 1, 1, RAGGED>(q, s);
    case 3: return many_rows(q) ? launch_ln_many<KIND, 3, RAGGED>(q, s)
                                : launch_ring<KIND, 4, 3, 16, 2, 1, RAGGED>(q, s);
    case 4: return many_rows(q) ? launch_ln_many<KIND, 4, RAGGED>(q, s)
                                : launch_ring<KIND, 4, 4, 16, 2, 1, RAGGED>(q, s);
    case 5: return launch_ring<KIND, 4, 5, 8, 2, 2, RAGGED>(q, s);
    case 6: return launch_ring<KIND, 4, 6, 8, 2, 2, RAGGED>(q, s);
    case 7: return launch_ring<KIND, 4, 7, 8, 2, 2, RAGGED>(q, s);
    default: return launch_ring<KIND, 4, 8, 8, 2, 2, RAGGED>(q, s);
    }
}

} // namespace

} // namespace dan
