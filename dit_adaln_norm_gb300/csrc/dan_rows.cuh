// dan_rows.cuh -- fused norm + adaLN modulate row kernels for sm_103a
// (included by dan_rows_rms.cu, dan_rows_gated.cu and dan_rows_ln.cu,
// which instantiate and launch them).
//
// RMSNorm ("SGLang diffusion fused-op package guide", section "Norm +
// scale/shift (adaLN)"; "PR #33854 report", key source excerpt) and
// LayerNorm without affine by Welford ("PR #34126 report", motivation
// section), each followed by the aten modulate chain
// y = bf16(bf16(n * bf16(1 + scale)) + shift).  The gated form first
// forms r' = bf16(r + bf16(gate * h)) and stores it.
//
// Design (HBM-bound row work, no tensor cores):
//  - One CTA per SM takes a contiguous block of rows.  Its producer thread
//    streams the rows into a ring of shared-memory slots with TMA bulk
//    copies (cp.async.bulk, completion counted on mbarriers, see
//    dan_ring.cuh), in row order, about eight rows ahead; consumer warps
//    take one row each, copy it from the slot into registers, release the
//    slot and compute while later rows are in flight.  Each row is read
//    from HBM once.
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
//    adjacent-pair tree padded with +0.  A consumer warp carries all D/2048
//    logical warps of its row.
//  - LayerNorm: 128 logical threads (four logical warps in one consumer
//    warp), thread t owns fragments t + 128k; Welford per element with
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
    int64_t rows;
    int64_t T;
    int64_t vs8; // batch stride of the vectors in 16-byte fragments
    int Bs;      // batches staged in shared memory; 0 = read vectors from global
    int F;       // fragments per row (D / 8)
    float eps;
    unsigned *status;            // device status word (bounded-wait failures)
    unsigned long long limit_ns; // bound of every wait
    unsigned *cta_status;        // per-CTA failure records (CTA_STATUS kernels only)
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

// Canonical sum of squares, rstd, normalise, modulate and store for one
// row whose fragments are in v (for the gated form v already holds r').
template <int LW, int NV, bool HAS_W, bool STAGED>
__device__ __forceinline__ void rms_row(const uint4 (&v)[LW][8], const RowParams &p, int64_t row,
                                        const uint4 *s_w, const uint4 *s_vec, int lane)
{
    constexpr int TPR = 32 * LW, F = 8 * TPR, D = 8 * F;
    constexpr int P2 = LW <= 1 ? 1 : LW <= 2 ? 2 : 4;
    constexpr int NP = LW / 2; // packed chain pairs per lane
    const int64_t bidx = row / p.T;

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
                    const float2 x2 = make_float2(elem(v[2 * q][k], e), elem(v[2 * q + 1][k], e));
                    acc2[q] = addmul2(acc2[q], x2, x2);
                }
                if (LW & 1) {
                    const float xv = elem(v[LW - 1][k], e);
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
    // Adjacent-pair tree over the 32 lanes of each logical warp, then over
    // the logical warp sums padded with +0.
#pragma unroll
    for (int off = 1; off < 32; off <<= 1)
#pragma unroll
        for (int j = 0; j < LW; ++j) acc[j] = __fadd_rn(acc[j], __shfl_xor_sync(kFull, acc[j], off));
    float t[P2];
#pragma unroll
    for (int k = 0; k < P2; ++k) t[k] = k < LW ? acc[k] : 0.0f;
#pragma unroll
    for (int off = 1; off < P2; off <<= 1)
#pragma unroll
        for (int k = 0; k < P2; k += 2 * off) t[k] = __fadd_rn(t[k], t[k + off]);
    const float2 rstd2 = dup2(defined_rsqrt(__fadd_rn(__fdiv_rn(t[0], (float)D), p.eps)));

#pragma unroll
    for (int j = 0; j < LW; ++j)
#pragma unroll
        for (int k = 0; k < 8; ++k) {
            const int f = rms_frag<LW>(j, k, lane);
            const uint4 o = vec_frag<NV, STAGED>(p, s_vec, bidx, f, 0);
            const uint4 sh = vec_frag<NV, STAGED>(p, s_vec, bidx, f, 1);
            uint4 wv = make_uint4(0, 0, 0, 0);
            if (HAS_W) wv = s_w[f];
            uint4 out;
#pragma unroll
            for (int w = 0; w < 4; ++w) {
                float2 t2 = mul2(wide2(word(v[j][k], w)), rstd2);
                if (HAS_W) t2 = mul2(t2, wide2(word(wv, w)));
                set_word(out, w, modulate_word(pack_bf16(t2.x, t2.y), word(o, w), word(sh, w)));
            }
            st_stream(p.y + row * F + f, out);
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

// One LayerNorm row (4 logical warps in one physical warp): statistics in
// the canonical Welford order, then normalise, modulate and store.
template <int FPT, bool RAGGED, bool STAGED>
__device__ __forceinline__ void ln_row(const uint4 (&v)[4][FPT], const RowParams &p, int64_t row,
                                       const InvTable2 &inv, const uint4 *s_vec, int lane)
{
    constexpr int NV = 2;
    const int F = p.F;
    const int64_t bidx = row / p.T;
    float wmean[4], wm2[4]; // per logical warp, folded over its 32 threads

    if (!RAGGED) {
        // Every logical thread holds FPT full fragments: counts are equal
        // everywhere, so each combine has c = 1/2 exactly.
        float2 mean2[2], m22[2];
#pragma unroll
        for (int q = 0; q < 2; ++q) mean2[q] = m22[q] = make_float2(0.0f, 0.0f);
#pragma unroll
        for (int k = 0; k < FPT; ++k)
#pragma unroll
            for (int e = 0; e < 8; ++e) {
                const float2 r = inv.v[8 * k + e + 1];
#pragma unroll
                for (int q = 0; q < 2; ++q) {
                    const float2 x2 = make_float2(elem(v[2 * q][k], e), elem(v[2 * q + 1][k], e));
                    const float2 d = sub2(x2, mean2[q]);
                    mean2[q] = addmul2(mean2[q], d, r);
                    m22[q] = addmul2(m22[q], d, sub2(x2, mean2[q]));
                }
            }
        float nA = (float)(8 * FPT);
#pragma unroll
        for (int off = 16; off >= 1; off >>= 1) {
#pragma unroll
            for (int q = 0; q < 2; ++q) {
                const float2 mb = make_float2(__shfl_down_sync(kFull, mean2[q].x, off),
                                              __shfl_down_sync(kFull, mean2[q].y, off));
                const float2 m2b = make_float2(__shfl_down_sync(kFull, m22[q].x, off),
                                               __shfl_down_sync(kFull, m22[q].y, off));
                combine_eq2(mean2[q], m22[q], mb, m2b, nA);
            }
            nA = 2.0f * nA;
        }
#pragma unroll
        for (int q = 0; q < 2; ++q) {
            wmean[2 * q] = __shfl_sync(kFull, mean2[q].x, 0);
            wmean[2 * q + 1] = __shfl_sync(kFull, mean2[q].y, 0);
            wm2[2 * q] = __shfl_sync(kFull, m22[q].x, 0);
            wm2[2 * q + 1] = __shfl_sync(kFull, m22[q].y, 0);
        }
    } else {
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            float mean = 0.0f, m2 = 0.0f;
            int nfr = 0;
#pragma unroll
            for (int k = 0; k < FPT; ++k) {
                if (ln_frag(j, lane, k) < F) {
                    nfr = k + 1;
#pragma unroll
                    for (int e = 0; e < 8; ++e) {
                        const float xv = elem(v[j][k], e);
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
    float mean, m2;
    if (!RAGGED) {
        const float nw = (float)(256 * FPT); // count of one logical warp
        float2 m01 = make_float2(wmean[0], wmean[1]), q01 = make_float2(wm2[0], wm2[1]);
        combine_eq2(m01, q01, make_float2(wmean[2], wmean[3]), make_float2(wm2[2], wm2[3]), nw);
        mean = m01.x;
        m2 = q01.x;
        combine_eq1(mean, m2, m01.y, q01.y, 2.0f * nw);
    } else {
        float N[4];
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            int cnt = 0; // 8 per valid fragment of the logical warp's threads
            for (int t = 32 * j; t < 32 * j + 32; ++t)
                for (int k = 0; k < FPT; ++k) cnt += (t + 128 * k < F) ? 8 : 0;
            N[j] = (float)cnt;
        }
        const Welford S =
            combine(combine(Welford{N[0], wmean[0], wm2[0]}, Welford{N[2], wmean[2], wm2[2]}),
                    combine(Welford{N[1], wmean[1], wm2[1]}, Welford{N[3], wmean[3], wm2[3]}));
        mean = S.mean;
        m2 = S.m2;
    }
    const float2 rstd2 = dup2(defined_rsqrt(__fadd_rn(__fdiv_rn(m2, (float)(8 * F)), p.eps)));
    const float2 mean2 = dup2(mean);

#pragma unroll
    for (int j = 0; j < 4; ++j)
#pragma unroll
        for (int k = 0; k < FPT; ++k) {
            const int f = ln_frag(j, lane, k);
            if (RAGGED && f >= F) continue;
            const uint4 o = vec_frag<NV, STAGED>(p, s_vec, bidx, f, 0);
            const uint4 sh = vec_frag<NV, STAGED>(p, s_vec, bidx, f, 1);
            uint4 out;
#pragma unroll
            for (int w = 0; w < 4; ++w) {
                const float2 t2 = mul2(sub2(wide2(word(v[j][k], w)), mean2), rstd2);
                set_word(out, w, modulate_word(pack_bf16(t2.x, t2.y), word(o, w), word(sh, w)));
            }
            st_stream(p.y + row * F + f, out);
        }
}

// ------------------------------------------------------- the ring kernel

enum RowKind { kRms = 0, kGated = 1, kLn = 2 };

// Shared memory: NW * SPC row slots (NIN inputs of D bf16 each; warp c
// owns slots c*SPC .. c*SPC+SPC-1), the norm weight, the staged vectors,
// then one mbarrier per slot.
template <int KIND>
struct RowShape {
    static constexpr int NIN = KIND == kGated ? 2 : 1; // bulk-copied inputs per row
    static constexpr int NV = KIND == kGated ? 3 : 2;  // staged vectors per batch
};

// CTA c takes the contiguous rows [c*R/G, (c+1)*R/G); its warp w takes the
// CTA's rows w, w + NW, w + 2NW, ... one at a time, the whole row in
// registers (LW logical warps per lane for RMS, 4 for LayerNorm), and
// requests each row SPC rows ahead into its own slots (dan_ring.cuh).
// CTA_STATUS kernels also keep one failure record per CTA in
// p.cta_status[blockIdx.x], cleared when the CTA starts.
template <int KIND, int LW, int FPT, int NW, int SPC, bool HAS_W, bool RAGGED, bool STAGED,
          bool CTA_STATUS = false>
__global__ void __launch_bounds__(32 * NW, 1)
    row_ring_kernel(const RowParams p, const InvTable2 inv)
{
    using Shape = RowShape<KIND>;
    using Pipe = WarpPipe<SPC>;
    constexpr int NIN = Shape::NIN, NV = Shape::NV;
    const int F = p.F;
    const unsigned row_bytes = (unsigned)F * 16u;

    extern __shared__ __align__(128) uint4 smem[];
    uint4 *ring = smem;                                 // NW * SPC * NIN * F
    uint4 *s_w = ring + (int64_t)NW * SPC * NIN * F;    // F if HAS_W
    uint4 *s_vec = s_w + (HAS_W ? F : 0);               // Bs * NV * F
    uint64_t *full = reinterpret_cast<uint64_t *>(s_vec + (int64_t)p.Bs * NV * F);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int64_t G = gridDim.x;
    const int64_t r0 = (int64_t)blockIdx.x * p.rows / G;
    const int n = (int)((int64_t)(blockIdx.x + 1) * p.rows / G - r0);

    if (threadIdx.x == 0) {
        for (int s = 0; s < NW * SPC; ++s) mbar_init(full + s, 1);
        mbar_init_fence();
    }
    grid_dependency_wait(); // no global access above this line
    allow_dependents();
    if (CTA_STATUS && threadIdx.x == 0) p.cta_status[blockIdx.x] = 0u;
    stage_begin<NV, HAS_W>(p, s_w, s_vec);
    __syncthreads(); // barriers initialised

    uint4 *slots = ring + (int64_t)warp * SPC * NIN * F;
    uint64_t *bar = full + warp * SPC;
    const int units = warp < n ? (n - warp + NW - 1) / NW : 0; // rows of this warp
    auto request = [&](int i) {                                // lane 0 only
        const int64_t row = r0 + warp + (int64_t)NW * i;
        uint4 *dst = slots + (int64_t)Pipe::slot(i) * NIN * F;
        uint64_t *b = bar + Pipe::slot(i);
        mbar_arrive_expect_tx(b, NIN * row_bytes);
        bulk_load(dst, p.x + row * F, row_bytes, b);
        if (NIN == 2) bulk_load(dst + F, p.h + row * F, row_bytes, b);
    };
    // The first SPC rows go out before waiting for the staged vectors.
    if (lane == 0)
        for (int i = 0; i < SPC && i < units; ++i) request(i);
    stage_end<NV>(p, s_vec);

    for (int i = 0; i < units; ++i) {
        if (!Pipe::wait(bar, i, p.limit_ns)) {
            const unsigned bits = Pipe::abort(bar, i, units, p.status, p.limit_ns);
            if (CTA_STATUS) set_status(p.cta_status + blockIdx.x, bits);
            return;
        }
        const uint4 *src = slots + (int64_t)Pipe::slot(i) * NIN * F;
        const int64_t row = r0 + warp + (int64_t)NW * i;
        if (KIND == kLn) {
            uint4 v[4][FPT];
#pragma unroll
            for (int j = 0; j < 4; ++j)
#pragma unroll
                for (int q = 0; q < FPT; ++q) {
                    const int f = ln_frag(j, lane, q);
                    v[j][q] = (!RAGGED || f < F) ? src[f] : make_uint4(0, 0, 0, 0);
                }
            slot_reads_done();
            if (lane == 0 && i + SPC < units) request(i + SPC);
            ln_row<FPT, RAGGED, STAGED>(v, p, row, inv, s_vec, lane);
        } else {
            uint4 v[LW][8];
            const int64_t bidx = row / p.T;
#pragma unroll
            for (int j = 0; j < LW; ++j)
#pragma unroll
                for (int q = 0; q < 8; ++q) {
                    const int f = rms_frag<LW>(j, q, lane);
                    v[j][q] = src[f];
                    if (KIND == kGated) { // r' = bf16(r + bf16(gate * h))
                        const uint4 g = vec_frag<NV, STAGED>(p, s_vec, bidx, f, 2);
                        const uint4 hh = src[F + f];
                        uint4 &r = v[j][q];
                        r = make_uint4(gated_word(r.x, g.x, hh.x), gated_word(r.y, g.y, hh.y),
                                       gated_word(r.z, g.z, hh.z), gated_word(r.w, g.w, hh.w));
                    }
                }
            slot_reads_done();
            if (lane == 0 && i + SPC < units) request(i + SPC);
            if (KIND == kGated)
#pragma unroll
                for (int j = 0; j < LW; ++j)
#pragma unroll
                    for (int q = 0; q < 8; ++q)
                        st_stream(p.r_out + row * F + rms_frag<LW>(j, q, lane), v[j][q]);
            rms_row<LW, NV, HAS_W, STAGED>(v, p, row, s_w, s_vec, lane);
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
    p.rows = q.B * q.T;
    p.T = q.T;
    p.vs8 = q.vs / 8;
    p.F = (int)(q.D / 8);
    p.eps = q.eps;
    p.Bs = 0;
    p.status = device_status();
    p.limit_ns = kWaitLimitNs;
    p.cta_status = nullptr;
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

// Shared memory a launch of row_ring_kernel<KIND, ..., NW, SPC> needs, with
// p.Bs set to the number of batches whose vectors are staged (all of them
// when they fit in the staging budget, else none).
template <int KIND, int NW, int SPC>
int ring_smem(const RowProblem &q, RowParams &p)
{
    using Shape = RowShape<KIND>;
    const int64_t row_bytes = q.D * 2;
    const int64_t fixed = (int64_t)NW * SPC * Shape::NIN * row_bytes +
                          (KIND != kLn && q.weight ? row_bytes : 0) + NW * SPC * 8;
    const int64_t vec_bytes = q.B * Shape::NV * row_bytes;
    const int64_t room = (int64_t)max_smem_optin() - fixed;
    p.Bs = (vec_bytes <= kStageBudget && vec_bytes <= room) ? (int)q.B : 0;
    return (int)(fixed + (p.Bs ? vec_bytes : 0));
}

// One CTA per SM (the slots and the warps' registers fill it), at most one
// per row; each CTA takes a contiguous block of rows.  `cta_status` is the
// per-CTA failure record array of CTA_STATUS kernels (nullptr otherwise).
template <int KIND, int LW, int FPT, int NW, int SPC, bool RAGGED, bool CTA_STATUS = false>
cudaError_t launch_ring(const RowProblem &q, cudaStream_t s, unsigned *cta_status = nullptr)
{
    RowParams p = make_params(q);
    p.cta_status = cta_status;
    const bool has_w = KIND != kLn && q.weight != nullptr;
    const int smem = ring_smem<KIND, NW, SPC>(q, p);
    const int grid = (int)(p.rows < sm_count() ? p.rows : sm_count());
    const InvTable2 inv = inv_table();
    auto go = [&](auto fn) -> cudaError_t {
        const cudaError_t e = allow_smem(fn, smem);
        if (e != cudaSuccess) return e;
        return launch_overlapped(fn, grid, 32 * NW, smem, s, p, inv);
    };
    constexpr bool CS = CTA_STATUS;
    if (has_w)
        return p.Bs ? go(row_ring_kernel<KIND, LW, FPT, NW, SPC, true, RAGGED, true, CS>)
                    : go(row_ring_kernel<KIND, LW, FPT, NW, SPC, true, RAGGED, false, CS>);
    return p.Bs ? go(row_ring_kernel<KIND, LW, FPT, NW, SPC, false, RAGGED, true, CS>)
                : go(row_ring_kernel<KIND, LW, FPT, NW, SPC, false, RAGGED, false, CS>);
}

template <bool RAGGED>
cudaError_t launch_ln_fpt(const RowProblem &q, cudaStream_t s)
{
    switch ((q.D + 1023) / 1024) {
    case 1: return launch_ring<kLn, 4, 1, 8, 1, RAGGED>(q, s);
    case 2: return launch_ring<kLn, 4, 2, 8, 1, RAGGED>(q, s);
    case 3: return launch_ring<kLn, 4, 3, 8, 1, RAGGED>(q, s);
    case 4: return launch_ring<kLn, 4, 4, 8, 1, RAGGED>(q, s);
    case 5: return launch_ring<kLn, 4, 5, 8, 1, RAGGED>(q, s);
    case 6: return launch_ring<kLn, 4, 6, 8, 1, RAGGED>(q, s);
    case 7: return launch_ring<kLn, 4, 7, 8, 1, RAGGED>(q, s);
    default: return launch_ring<kLn, 4, 8, 8, 1, RAGGED>(q, s);
    }
}

} // namespace

} // namespace dan
