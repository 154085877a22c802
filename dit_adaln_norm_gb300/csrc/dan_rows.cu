// dan_rows.cu -- fused norm + adaLN modulate row kernels for sm_103a.
//
// RMSNorm ("SGLang diffusion fused-op package guide", section "Norm +
// scale/shift (adaLN)"; "PR #33854 report", key source excerpt) and
// LayerNorm without affine by Welford ("PR #34126 report", motivation
// section), each followed by the aten modulate chain
// y = bf16(bf16(n * bf16(1 + scale)) + shift).  The gated form first
// forms r' = bf16(r + bf16(gate * h)) and stores it.
//
// Design (HBM-bound row work, no tensor cores):
//  - Persistent grid: SMs x resident CTAs.  CTA c takes rows c, c + G,
//    c + 2G, ... (G = grid size); its row slots (one or more warps each)
//    take those rows in turn.  The arithmetic of a row depends only on the
//    row's columns, never on which warp, CTA or launch computes it, so the
//    output bits are independent of B, T and the grid (batch invariance).
//  - A row is loaded once into registers with 16-byte coalesced loads (one
//    warp instruction moves 512 contiguous bytes), reduced, normalised,
//    modulated and stored; it is never re-read.
//  - bf16(1 + scale), shift, gate and the norm weight are staged in shared
//    memory once per CTA for every batch (when they fit), so the per-element
//    work reads them with conflict-free 16-byte shared loads.  The staging
//    copies are issued before the first rows' loads and completed after
//    them, so the two overlap.
//  - Canonical RMS order: logical thread tx (TPR = D/64 of them) owns the
//    fragments TPR*b + tx (b = 0..7) as one sequential chain; lanes fold by
//    the butterfly (= the adjacent-pair tree); logical warp sums fold by the
//    adjacent-pair tree padded with +0.  A physical warp carries LW logical
//    warps; PW physical warps share a row through shared memory.
//  - LayerNorm: 128 logical threads, thread t owns fragments t + 128k;
//    Welford per element with rn(1/n) from a host-computed table; warps fold
//    by an ordered xor butterfly that reproduces the shfl.down tree in every
//    lane; the four warp states fold as (W0 + W2) + (W1 + W3).
#include "dan_device.cuh"
#include "dan_internal.h"

#include <mutex>
#include <unordered_map>

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
    int64_t rows;
    int64_t T;
    int64_t vs8; // batch stride of the vectors in 16-byte fragments
    int Bs;      // batches staged in shared memory; 0 = read vectors from global
    int F;       // fragments per row (D / 8)
    float eps;
};

__device__ __forceinline__ void named_barrier(int id, int threads)
{
    asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(threads) : "memory");
}

// Per-batch vector fragment f: which = 0 -> bf16(1 + scale), 1 -> shift,
// 2 -> gate.  Staged copy when available, else computed from global.
template <int NV>
__device__ __forceinline__ uint4 vec_frag(const RowParams &p, const uint4 *s_vec, int64_t b, int f,
                                          int which)
{
    if (p.Bs) return s_vec[(b * NV + which) * p.F + f];
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

template <int LW, int PW, bool GATED>
struct RmsRow {
    uint4 v[LW][8];
    uint4 h[GATED ? LW : 1][8];
};

// Issue the 16-byte loads of one row (x, and h for the gated form).
template <int LW, int PW, bool GATED>
__device__ __forceinline__ void rms_load(RmsRow<LW, PW, GATED> &b, const RowParams &p, int64_t row,
                                         int pw, int lane)
{
    constexpr int TPR = 32 * LW * PW, F = 8 * TPR;
#pragma unroll
    for (int j = 0; j < LW; ++j)
#pragma unroll
        for (int k = 0; k < 8; ++k) {
            const int f = TPR * k + 32 * (pw * LW + j) + lane;
            b.v[j][k] = ld_stream(p.x + row * F + f);
            if (GATED) b.h[j][k] = ld_stream(p.h + row * F + f);
        }
}

// Gated residual (stored), canonical sum of squares, rstd, normalise,
// modulate and store for one row whose data is in `b`.
template <int LW, int PW, int WARPS, bool GATED, bool HAS_W>
__device__ __forceinline__ void rms_process(RmsRow<LW, PW, GATED> &b, const RowParams &p,
                                            int64_t row, const uint4 *s_w, const uint4 *s_vec,
                                            float *s_red, int slot, int pw, int lane, int &parity)
{
    constexpr int WPR = LW * PW, TPR = 32 * WPR, F = 8 * TPR, D = 8 * F;
    constexpr int RS = WARPS / PW;
    constexpr int NV = GATED ? 3 : 2;
    constexpr int P2 = WPR <= 1 ? 1 : WPR <= 2 ? 2 : WPR <= 4 ? 4 : 8;
    constexpr int NP = LW / 2; // packed chain pairs per lane
    const int64_t bidx = row / p.T;

    if (GATED) { // r' = bf16(r + bf16(gate * h)), stored, then normalised
#pragma unroll
        for (int j = 0; j < LW; ++j)
#pragma unroll
            for (int k = 0; k < 8; ++k) {
                const int f = TPR * k + 32 * (pw * LW + j) + lane;
                const uint4 g = vec_frag<NV>(p, s_vec, bidx, f, 2);
                uint4 &r = b.v[j][k];
                const uint4 &hh = b.h[j][k];
                r = make_uint4(gated_word(r.x, g.x, hh.x), gated_word(r.y, g.y, hh.y),
                               gated_word(r.z, g.z, hh.z), gated_word(r.w, g.w, hh.w));
                st_stream(p.r_out + row * F + f, r);
            }
    }

    // Sum of squares: one ordered chain per logical thread (v fastest, then
    // the fragment index); logical threads j, j+1 of a lane share packed
    // multiplies.
    float acc[LW];
    {
        float2 acc2[NP > 0 ? NP : 1];
        float acc1 = 0.0f;
#pragma unroll
        for (int q = 0; q < NP; ++q) acc2[q] = make_float2(0.0f, 0.0f);
#pragma unroll
        for (int k = 0; k < 8; ++k)
#pragma unroll
            for (int e = 0; e < 8; ++e) {
#pragma unroll
                for (int q = 0; q < NP; ++q) {
                    const float2 x2 = make_float2(elem(b.v[2 * q][k], e), elem(b.v[2 * q + 1][k], e));
                    acc2[q] = addmul2(acc2[q], x2, x2);
                }
                if (LW & 1) {
                    const float xv = elem(b.v[LW - 1][k], e);
                    acc1 = __fadd_rn(acc1, __fmul_rn(xv, xv));
                }
            }
#pragma unroll
        for (int q = 0; q < NP; ++q) {
            acc[2 * q] = acc2[q].x;
            acc[2 * q + 1] = acc2[q].y;
        }
        if (LW & 1) acc[LW - 1] = acc1;
    }
    // Adjacent-pair tree over the 32 lanes of each logical warp.
#pragma unroll
    for (int off = 1; off < 32; off <<= 1)
#pragma unroll
        for (int j = 0; j < LW; ++j) acc[j] = __fadd_rn(acc[j], __shfl_xor_sync(kFull, acc[j], off));

    // Logical warp sums -> adjacent-pair tree padded with +0.
    float t[P2];
#pragma unroll
    for (int k = 0; k < P2; ++k) t[k] = 0.0f;
    if (PW == 1) {
#pragma unroll
        for (int j = 0; j < LW; ++j) t[j] = acc[j];
    } else {
        float *red = s_red + (parity * RS + slot) * WPR;
        if (lane == 0)
#pragma unroll
            for (int j = 0; j < LW; ++j) red[pw * LW + j] = acc[j];
        named_barrier(1 + slot, PW * 32);
#pragma unroll
        for (int k = 0; k < WPR; ++k) t[k] = red[k];
        parity ^= 1;
    }
#pragma unroll
    for (int off = 1; off < P2; off <<= 1)
#pragma unroll
        for (int k = 0; k < P2; k += 2 * off) t[k] = __fadd_rn(t[k], t[k + off]);
    const float2 rstd2 = dup2(defined_rsqrt(__fadd_rn(__fdiv_rn(t[0], (float)D), p.eps)));

#pragma unroll
    for (int j = 0; j < LW; ++j)
#pragma unroll
        for (int k = 0; k < 8; ++k) {
            const int f = TPR * k + 32 * (pw * LW + j) + lane;
            const uint4 o = vec_frag<NV>(p, s_vec, bidx, f, 0);
            const uint4 sh = vec_frag<NV>(p, s_vec, bidx, f, 1);
            uint4 wv = make_uint4(0, 0, 0, 0);
            if (HAS_W) wv = s_w[f];
            uint4 out;
#pragma unroll
            for (int w = 0; w < 4; ++w) {
                float2 t2 = mul2(wide2(word(b.v[j][k], w)), rstd2);
                if (HAS_W) t2 = mul2(t2, wide2(word(wv, w)));
                set_word(out, w, modulate_word(pack_bf16(t2.x, t2.y), word(o, w), word(sh, w)));
            }
            st_stream(p.y + row * F + f, out);
        }
}

// Rows of a CTA are blockIdx.x + G*i (G = grid size); row slot s takes
// i = s, s + RS, s + 2RS, ...  Two register buffers alternate: the loads of
// a slot's next row are issued before its current row is processed, so
// each warp keeps up to two rows in flight.
template <int LW, int PW, int WARPS, int MINB, bool GATED, bool HAS_W>
__global__ void __launch_bounds__(WARPS * 32, MINB)
    rms_modulate_kernel(const RowParams p)
{
    constexpr int TPR = 32 * LW * PW, F = 8 * TPR;
    constexpr int RS = WARPS / PW;
    constexpr int NV = GATED ? 3 : 2;

    extern __shared__ uint4 smem[];
    uint4 *s_w = smem;
    uint4 *s_vec = smem + (HAS_W ? F : 0);
    float *s_red = reinterpret_cast<float *>(s_vec + (int64_t)p.Bs * NV * F);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int slot = warp / PW, pw = warp - slot * PW;
    const int64_t step = (int64_t)gridDim.x * RS;

    RmsRow<LW, PW, GATED> A, B;
    int64_t ra = blockIdx.x + (int64_t)gridDim.x * slot, rb = ra + step;
    stage_begin<NV, HAS_W>(p, s_w, s_vec);
    if (ra < p.rows) rms_load(A, p, ra, pw, lane);
    if (rb < p.rows) rms_load(B, p, rb, pw, lane);
    stage_end<NV>(p, s_vec);

    int parity = 0;
    while (ra < p.rows) {
        rms_process<LW, PW, WARPS, GATED, HAS_W>(A, p, ra, s_w, s_vec, s_red, slot, pw, lane,
                                                 parity);
        ra = rb + step;
        if (ra < p.rows) rms_load(A, p, ra, pw, lane);
        if (rb >= p.rows) break;
        rms_process<LW, PW, WARPS, GATED, HAS_W>(B, p, rb, s_w, s_vec, s_red, slot, pw, lane,
                                                 parity);
        rb = ra + step;
        if (rb < p.rows) rms_load(B, p, rb, pw, lane);
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

template <int LW, int FPT>
struct LnRow {
    uint4 v[LW][FPT];
};

// fragment index of logical thread (warp pw, chain j, lane), k-th visit
template <int LW>
__device__ __forceinline__ int ln_frag(int pw, int j, int lane, int k)
{
    return 32 * (pw * LW + j) + lane + 128 * k;
}

template <int LW, int FPT, bool RAGGED>
__device__ __forceinline__ void ln_load(LnRow<LW, FPT> &b, const RowParams &p, int64_t row, int pw,
                                        int lane)
{
    const int F = p.F;
#pragma unroll
    for (int j = 0; j < LW; ++j)
#pragma unroll
        for (int k = 0; k < FPT; ++k) {
            const int f = ln_frag<LW>(pw, j, lane, k);
            b.v[j][k] = (!RAGGED || f < F) ? ld_stream(p.x + row * F + f) : make_uint4(0, 0, 0, 0);
        }
}

template <int LW, int PW, int FPT, bool RAGGED, int WARPS>
__device__ __forceinline__ void ln_process(LnRow<LW, FPT> &b, const RowParams &p, int64_t row,
                                           const InvTable2 &inv, const uint4 *s_vec, float *s_red,
                                           int slot, int pw, int lane, int &parity)
{
    constexpr int RS = WARPS / PW;
    constexpr int NV = 2;
    constexpr int NQ = LW / 2; // packed chain pairs per lane (LW is 2 or 4)
    const int F = p.F;
    const int64_t bidx = row / p.T;
    // Statistics of the lane's logical warps: (mean, m2) of logical warp
    // pw*LW + j, already folded over its 32 threads.
    float wmean[LW], wm2[LW];

    if (!RAGGED) {
        // Every logical thread holds FPT full fragments: counts are equal
        // everywhere, so each combine has c = 1/2 exactly.
        float2 mean2[NQ], m22[NQ];
#pragma unroll
        for (int q = 0; q < NQ; ++q) mean2[q] = m22[q] = make_float2(0.0f, 0.0f);
#pragma unroll
        for (int k = 0; k < FPT; ++k)
#pragma unroll
            for (int e = 0; e < 8; ++e) {
                const float2 r = inv.v[8 * k + e + 1];
#pragma unroll
                for (int q = 0; q < NQ; ++q) {
                    const float2 x2 = make_float2(elem(b.v[2 * q][k], e), elem(b.v[2 * q + 1][k], e));
                    const float2 d = sub2(x2, mean2[q]);
                    mean2[q] = addmul2(mean2[q], d, r);
                    m22[q] = addmul2(m22[q], d, sub2(x2, mean2[q]));
                }
            }
        float nA = (float)(8 * FPT);
#pragma unroll
        for (int off = 16; off >= 1; off >>= 1) {
#pragma unroll
            for (int q = 0; q < NQ; ++q) {
                const float2 mb = make_float2(__shfl_down_sync(kFull, mean2[q].x, off),
                                              __shfl_down_sync(kFull, mean2[q].y, off));
                const float2 m2b = make_float2(__shfl_down_sync(kFull, m22[q].x, off),
                                               __shfl_down_sync(kFull, m22[q].y, off));
                combine_eq2(mean2[q], m22[q], mb, m2b, nA);
            }
            nA = 2.0f * nA;
        }
#pragma unroll
        for (int q = 0; q < NQ; ++q) {
            wmean[2 * q] = __shfl_sync(kFull, mean2[q].x, 0);
            wmean[2 * q + 1] = __shfl_sync(kFull, mean2[q].y, 0);
            wm2[2 * q] = __shfl_sync(kFull, m22[q].x, 0);
            wm2[2 * q + 1] = __shfl_sync(kFull, m22[q].y, 0);
        }
    } else {
#pragma unroll
        for (int j = 0; j < LW; ++j) {
            float mean = 0.0f, m2 = 0.0f;
            int nfr = 0;
#pragma unroll
            for (int k = 0; k < FPT; ++k) {
                if (ln_frag<LW>(pw, j, lane, k) < F) {
                    nfr = k + 1;
#pragma unroll
                    for (int e = 0; e < 8; ++e) {
                        const float xv = elem(b.v[j][k], e);
                        const float d = __fsub_rn(xv, mean);
                        mean = __fadd_rn(mean, __fmul_rn(d, inv.v[8 * k + e + 1].x));
                        m2 = __fadd_rn(m2, __fmul_rn(d, __fsub_rn(xv, mean)));
                    }
                }
            }
            Welford st{(float)(8 * nfr), mean, m2};
            st = warp_fold(st, lane);
            wmean[j] = st.mean;
            wm2[j] = st.m2;
        }
    }

    // The four logical warps: (W0 + W2) + (W1 + W3).
    float M[4], Q[4];
    if (PW == 1) {
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            M[j] = wmean[j];
            Q[j] = wm2[j];
        }
    } else {
        float *red = s_red + (parity * RS + slot) * 8;
        if (lane == 0)
#pragma unroll
            for (int j = 0; j < LW; ++j) {
                red[2 * (pw * LW + j) + 0] = wmean[j];
                red[2 * (pw * LW + j) + 1] = wm2[j];
            }
        named_barrier(1 + slot, PW * 32);
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            M[j] = red[2 * j];
            Q[j] = red[2 * j + 1];
        }
        parity ^= 1;
    }
    float mean, m2;
    if (!RAGGED) {
        const float nw = (float)(256 * FPT); // count of one logical warp
        float2 m01 = make_float2(M[0], M[1]), q01 = make_float2(Q[0], Q[1]);
        combine_eq2(m01, q01, make_float2(M[2], M[3]), make_float2(Q[2], Q[3]), nw);
        mean = m01.x;
        m2 = q01.x;
        combine_eq1(mean, m2, m01.y, q01.y, 2.0f * nw);
    } else {
        float N[4];
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            // count of logical warp j: 8 per valid fragment of its threads
            int cnt = 0;
            for (int t = 32 * j; t < 32 * j + 32; ++t)
                for (int k = 0; k < FPT; ++k) cnt += (t + 128 * k < F) ? 8 : 0;
            N[j] = (float)cnt;
        }
        const Welford S = combine(combine(Welford{N[0], M[0], Q[0]}, Welford{N[2], M[2], Q[2]}),
                                  combine(Welford{N[1], M[1], Q[1]}, Welford{N[3], M[3], Q[3]}));
        mean = S.mean;
        m2 = S.m2;
    }
    const float2 rstd2 = dup2(defined_rsqrt(__fadd_rn(__fdiv_rn(m2, (float)(8 * F)), p.eps)));
    const float2 mean2 = dup2(mean);

#pragma unroll
    for (int j = 0; j < LW; ++j)
#pragma unroll
        for (int k = 0; k < FPT; ++k) {
            const int f = ln_frag<LW>(pw, j, lane, k);
            if (RAGGED && f >= F) continue;
            const uint4 o = vec_frag<NV>(p, s_vec, bidx, f, 0);
            const uint4 sh = vec_frag<NV>(p, s_vec, bidx, f, 1);
            uint4 out;
#pragma unroll
            for (int w = 0; w < 4; ++w) {
                const float2 t2 = mul2(sub2(wide2(word(b.v[j][k], w)), mean2), rstd2);
                set_word(out, w, modulate_word(pack_bf16(t2.x, t2.y), word(o, w), word(sh, w)));
            }
            st_stream(p.y + row * F + f, out);
        }
}

// Same row schedule and two-buffer pipeline as the RMS kernel.
template <int LW, int PW, int FPT, bool RAGGED, int WARPS, int MINB>
__global__ void __launch_bounds__(WARPS * 32, MINB)
    ln_modulate_kernel(const RowParams p, const InvTable2 inv)
{
    constexpr int RS = WARPS / PW;
    constexpr int NV = 2;

    extern __shared__ uint4 smem[];
    uint4 *s_vec = smem;
    float *s_red = reinterpret_cast<float *>(s_vec + (int64_t)p.Bs * NV * p.F);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int slot = warp / PW, pw = warp - slot * PW;
    const int64_t step = (int64_t)gridDim.x * RS;

    LnRow<LW, FPT> A, B;
    int64_t ra = blockIdx.x + (int64_t)gridDim.x * slot, rb = ra + step;
    stage_begin<NV, false>(p, nullptr, s_vec);
    if (ra < p.rows) ln_load<LW, FPT, RAGGED>(A, p, ra, pw, lane);
    if (rb < p.rows) ln_load<LW, FPT, RAGGED>(B, p, rb, pw, lane);
    stage_end<NV>(p, s_vec);

    int parity = 0;
    while (ra < p.rows) {
        ln_process<LW, PW, FPT, RAGGED, WARPS>(A, p, ra, inv, s_vec, s_red, slot, pw, lane, parity);
        ra = rb + step;
        if (ra < p.rows) ln_load<LW, FPT, RAGGED>(A, p, ra, pw, lane);
        if (rb >= p.rows) break;
        ln_process<LW, PW, FPT, RAGGED, WARPS>(B, p, rb, inv, s_vec, s_red, slot, pw, lane, parity);
        rb = ra + step;
        if (rb < p.rows) ln_load<LW, FPT, RAGGED>(B, p, rb, pw, lane);
    }
}

// ------------------------------------------------------------- launching

namespace {

// Largest shared-memory budget for staged vectors; beyond it the kernel
// reads them from global (identical arithmetic, e.g. thousands of batches).
constexpr int kStageBudget = 96 * 1024;

struct LaunchShape {
    int grid;
    int smem;
};

std::mutex g_mu;
std::unordered_map<const void *, int> g_smem_set; // kernel -> max dyn smem configured
std::unordered_map<uint64_t, int> g_occupancy;     // (device, kernel, smem) -> CTAs per SM

// Resident CTAs per SM for `fn` at this block/smem size (cached); sets the
// dynamic shared-memory limit the first time a kernel needs more than 48 KB.
template <typename K>
int resident_ctas(K fn, int threads, int smem)
{
    std::lock_guard<std::mutex> lk(g_mu);
    const void *key = reinterpret_cast<const void *>(fn);
    auto it = g_smem_set.find(key);
    if (smem > 48 * 1024 && (it == g_smem_set.end() || it->second < smem)) {
        cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
        g_smem_set[key] = smem;
    }
    int dev = 0;
    cudaGetDevice(&dev);
    const uint64_t okey = (reinterpret_cast<uint64_t>(key) * 1315423911u) ^
                          ((uint64_t)(unsigned)smem << 8) ^ (uint64_t)(unsigned)dev;
    auto oit = g_occupancy.find(okey);
    if (oit != g_occupancy.end()) return oit->second;
    int n = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, fn, threads, smem) != cudaSuccess || n < 1)
        n = 1;
    g_occupancy[okey] = n;
    return n;
}

RowParams make_params(const RowProblem &q, int nv)
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
    p.rows = q.B * q.T;
    p.T = q.T;
    p.vs8 = q.vs / 8;
    p.F = (int)(q.D / 8);
    p.eps = q.eps;
    const int64_t per_batch = (int64_t)nv * q.D * 2;
    p.Bs = (q.B * per_batch <= kStageBudget) ? (int)q.B : 0;
    return p;
}

template <typename K, typename... Args>
cudaError_t launch(K fn, int warps, int row_slots, const RowParams &p, int smem, cudaStream_t s,
                   Args... extra)
{
    const int threads = warps * 32;
    const int per_sm = resident_ctas(fn, threads, smem);
    const int64_t want = (p.rows + row_slots - 1) / row_slots;
    const int64_t cap = (int64_t)sm_count() * per_sm;
    const int grid = (int)(want < cap ? want : cap);
    fn<<<grid, threads, smem, s>>>(p, extra...);
    return cudaGetLastError();
}

template <int LW, int PW, int WARPS, int MINB, bool GATED>
cudaError_t launch_rms_t(const RowProblem &q, cudaStream_t s)
{
    constexpr int NV = GATED ? 3 : 2;
    const RowParams p = make_params(q, NV);
    const bool has_w = q.weight != nullptr;
    const int smem = (int)((has_w ? q.D * 2 : 0) + (int64_t)p.Bs * NV * q.D * 2 +
                           (PW > 1 ? 2 * (WARPS / PW) * LW * PW * 4 : 0));
    if (has_w)
        return launch(rms_modulate_kernel<LW, PW, WARPS, MINB, GATED, true>, WARPS, WARPS / PW, p,
                      smem, s);
    return launch(rms_modulate_kernel<LW, PW, WARPS, MINB, GATED, false>, WARPS, WARPS / PW, p,
                  smem, s);
}

template <int LW, int PW, int FPT, bool RAGGED>
cudaError_t launch_ln_t(const RowProblem &q, cudaStream_t s)
{
    // two row buffers of LW * FPT fragments: 12 warps per SM up to 4096
    constexpr int WARPS = FPT <= 2 ? 16 : 12;
    constexpr int MINB = 1;
    const RowParams p = make_params(q, 2);
    InvTable2 inv;
    inv.v[0] = make_float2(0.0f, 0.0f);
    for (int n = 1; n <= 64; ++n) {
        const float r = 1.0f / (float)n; // IEEE division on the host
        inv.v[n] = make_float2(r, r);
    }
    const int smem = (int)((int64_t)p.Bs * 2 * q.D * 2 + (PW > 1 ? 2 * (WARPS / PW) * 8 * 4 : 0));
    return launch(ln_modulate_kernel<LW, PW, FPT, RAGGED, WARPS, MINB>, WARPS, WARPS / PW, p, smem,
                  s, inv);
}

template <bool RAGGED>
cudaError_t launch_ln_fpt(const RowProblem &q, cudaStream_t s)
{
    switch ((q.D + 1023) / 1024) {
    case 1: return launch_ln_t<4, 1, 1, RAGGED>(q, s);
    case 2: return launch_ln_t<4, 1, 2, RAGGED>(q, s);
    case 3: return launch_ln_t<4, 1, 3, RAGGED>(q, s);
    case 4: return launch_ln_t<4, 1, 4, RAGGED>(q, s);
    case 5: return launch_ln_t<2, 2, 5, RAGGED>(q, s);
    case 6: return launch_ln_t<2, 2, 6, RAGGED>(q, s);
    case 7: return launch_ln_t<2, 2, 7, RAGGED>(q, s);
    default: return launch_ln_t<2, 2, 8, RAGGED>(q, s);
    }
}

} // namespace

// Configurations (logical warps per warp, warps per row, warps per CTA,
// CTAs per SM): chosen so that the two row buffers fit the register file.
cudaError_t launch_rms_modulate(const RowProblem &q, cudaStream_t s)
{
    switch (q.D) {
    case 2048: return launch_rms_t<1, 1, 8, 2, false>(q, s);
    case 4096: return launch_rms_t<2, 1, 12, 1, false>(q, s);
    case 6144: return launch_rms_t<1, 3, 12, 1, false>(q, s);
    default: return launch_rms_t<2, 2, 12, 1, false>(q, s); // 8192
    }
}

cudaError_t launch_gated_rms_modulate(const RowProblem &q, cudaStream_t s)
{
    switch (q.D) {
    case 2048: return launch_rms_t<1, 1, 8, 2, true>(q, s);
    case 4096: return launch_rms_t<1, 2, 12, 1, true>(q, s);
    case 6144: return launch_rms_t<1, 3, 12, 1, true>(q, s);
    default: return launch_rms_t<1, 4, 12, 1, true>(q, s); // 8192
    }
}

cudaError_t launch_ln_modulate(const RowProblem &q, cudaStream_t s)
{
    return (q.D % 1024) ? launch_ln_fpt<true>(q, s) : launch_ln_fpt<false>(q, s);
}

} // namespace dan
