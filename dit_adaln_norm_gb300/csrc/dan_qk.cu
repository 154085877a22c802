// dan_qk.cu -- QK-RMSNorm + RoPE + V copy epilogue for sm_103a.
//
// "PR #37123 report" (Qwen-Image FP8 QKV projection and Blackwell
// epilogue), implementation section 3: one kernel walks the Q/K/V work of
// the text and image token streams, normalises every head of Q and K with
// that stream's RMSNorm weight, rotates it with the stream's fp32 cos/sin
// row, copies V, and writes joint [text, image] buffers; inputs are
// zero-copy row-strided views of the packed QKV GEMM output (section 4).
// The page's kernel rotates interleaved pairs (is_neox=False) at head_dim
// 128; the same kernel also takes head_dim 64 and the neox rotation of
// halves, the QK-norm + RoPE variants the guide lists for other DiTs.
//
// Work unit = (token, Q|K|V, group of heads): one bulk copy into a
// shared-memory slot, processed by one warp (dan_ring.cuh).  LPH = HD/8
// lanes cover one head, lane fl owning the 16-byte fragment of columns
// 8fl..8fl+7, so each head is one coalesced load/store and the 32/LPH head
// slots of a warp take adjacent heads.  Head RMS: each lane's 8 squares in
// column order, then the adjacent-pair tree over the head's LPH lanes,
// done as a recursive-halving fold so that each lane ends with the sums of
// 16/LPH heads.
#include "dan_device.cuh"
#include "dan_internal.h"
#include "dan_ring.cuh"

namespace dan {

struct QkParams {
    const uint4 *q[2], *k[2], *v[2];
    int64_t T0;         // text tokens
    int64_t T_all;      // text + image tokens
    int64_t stride8[2]; // row stride in 16-byte fragments
    const uint4 *wq[2], *wk[2];
    const float4 *rope[2];
    float eps[2];
    uint4 *q_out, *k_out, *v_out;
    int H;
    int groups; // head groups per (token, kind)
    unsigned *status;
    unsigned long long limit_ns;
};

constexpr int kQkNW = 8;  // warps per CTA (measured best among 4..16)
constexpr int kQkPre = 3; // units per warp prefetched into L2 before the dependency wait
constexpr int kQkSPC = 3; // slots per warp (with the first units prefetched into L2 before the
                          // dependency wait: C5 26.02 us with two slots, 25.76 with three;
                          // 10 or 12 warps x 2 slots were slower)
constexpr int kHeadsPerLane = 12; // head fragments a lane holds per unit

// Shape of the work for head_dim HD.
template <int HD>
struct QkShape {
    static constexpr int LPH = HD / 8;             // lanes (and fragments) per head
    static constexpr int GPS = 32 / LPH;           // heads per warp step
    static constexpr int GROUP = kHeadsPerLane * GPS; // heads per unit
    static constexpr int DATA = GROUP * LPH;       // fragments of a unit's heads (6 KB)
    static constexpr int ROPE = HD / 4;            // fragments of a cos/sin row (HD fp32)
    static constexpr int SLOT = DATA + 32;         // slot: heads, then the cos/sin row
    static constexpr int LEVELS = LPH == 16 ? 4 : 3; // fold levels over the head's lanes
    static constexpr int NK = 16 >> LEVELS;        // head sums a lane ends with
};

// One unit of work = (token, Q|K|V, group of heads), as loaded registers:
// the head fragments plus, for Q and K, the weight fragment and the cos/sin
// of this lane's columns (interleaved: four pairs; neox: eight columns).
struct QkUnit {
    uint4 x[kHeadsPerLane];
    uint4 w;
    float4 c[2], s[2];
    int64_t tok;
    int kind, h0, s_;
};

// Unit k of CTA t0 (of G = gridDim.x, which takes the tokens t0, t0 + G,
// t0 + 2G, ...): token t0 + G * (k / (3 * groups)), then Q, K, V, each split
// in head groups of GROUP heads.
template <int HD>
__device__ __forceinline__ void qk_unit(QkUnit &U, const QkParams &p, int64_t t0, int k)
{
    if (p.groups == 1) { // one unit per (token, kind); k / 3 by a constant
        const unsigned uk = (unsigned)k;
        U.tok = t0 + (int64_t)gridDim.x * (uk / 3u);
        U.kind = (int)(uk % 3u);
        U.h0 = 0;
    } else {
        const int per_tok = 3 * p.groups;
        U.tok = t0 + (int64_t)gridDim.x * (k / per_tok);
        const int rem = k % per_tok;
        U.kind = rem / p.groups;
        U.h0 = (rem % p.groups) * QkShape<HD>::GROUP;
    }
    U.s_ = U.tok < p.T0 ? 0 : 1;
}

template <int HD>
__device__ __forceinline__ const uint4 *qk_src(const QkUnit &U, const QkParams &p)
{
    const int64_t t = U.s_ ? U.tok - p.T0 : U.tok;
    return (U.kind == 0 ? p.q[U.s_] : U.kind == 1 ? p.k[U.s_] : p.v[U.s_]) + t * p.stride8[U.s_] +
           U.h0 * QkShape<HD>::LPH;
}

template <int HD>
__device__ __forceinline__ int qk_heads(const QkUnit &U, const QkParams &p)
{
    constexpr int G = QkShape<HD>::GROUP;
    return p.H - U.h0 < G ? p.H - U.h0 : G;
}

template <int HD>
__device__ __forceinline__ const float4 *qk_rope_row(const QkUnit &U, const QkParams &p)
{
    const int64_t t = U.s_ ? U.tok - p.T0 : U.tok;
    return p.rope[U.s_] + t * QkShape<HD>::ROPE;
}

// Copy the unit's heads from its slot into registers, with, for Q and K,
// the stream's weight fragment (staged in s_w: wq_txt, wk_txt, wq_img,
// wk_img) and this lane's cos/sin (in the slot).
template <int HD, bool NEOX>
__device__ __forceinline__ void qk_take(QkUnit &U, const QkParams &p, const uint4 *slot,
                                        const uint4 *s_w, int hs, int fl)
{
    using S = QkShape<HD>;
    const int nh = qk_heads<HD>(U, p);
#pragma unroll
    for (int k = 0; k < kHeadsPerLane; ++k) {
        const int hh = hs + S::GPS * k;
        U.x[k] = hh < nh ? slot[hh * S::LPH + fl] : make_uint4(0, 0, 0, 0);
    }
    if (U.kind != 2) {
        U.w = s_w[(2 * U.s_ + U.kind) * S::LPH + fl];
        const float4 *rope = reinterpret_cast<const float4 *>(slot + S::DATA);
        if (NEOX) { // columns i = 8 (fl mod LPH/2) + e of the first half
            const int b = 2 * (fl % (S::LPH / 2));
            U.c[0] = rope[b];
            U.c[1] = rope[b + 1];
            U.s[0] = rope[S::ROPE / 2 + b];
            U.s[1] = rope[S::ROPE / 2 + b + 1];
        } else {                     // pairs 4fl .. 4fl+3
            U.c[0] = rope[fl];
            U.s[0] = rope[S::ROPE / 2 + fl];
        }
    }
}

// Reverse the low L bits of l.
template <int L>
__device__ __forceinline__ int brev(int l)
{
    int r = 0;
#pragma unroll
    for (int i = 0; i < L; ++i) r |= ((l >> i) & 1) << (L - 1 - i);
    return r;
}

__device__ __forceinline__ float f4(const float4 &v, int i)
{
    return i == 0 ? v.x : i == 1 ? v.y : i == 2 ? v.z : v.w;
}

template <int HD, bool NEOX>
__device__ __forceinline__ void qk_process(const QkUnit &U, const QkParams &p, int hs, int fl)
{
    using S = QkShape<HD>;
    uint4 *dst = (U.kind == 0 ? p.q_out : U.kind == 1 ? p.k_out : p.v_out) +
                 U.tok * p.H * S::LPH;
    if (U.kind == 2) { // V: bit copy
#pragma unroll
        for (int k = 0; k < kHeadsPerLane; ++k) {
            const int h = U.h0 + hs + S::GPS * k;
            if (h < p.H) st_stream(dst + h * S::LPH + fl, U.x[k]);
        }
        return;
    }

    // The lane's columns widened to fp32 once, as pairs of heads: x2[j][e]
    // holds column e of heads 2j and 2j+1, so the packed operations of the
    // squares and of the normalisation each serve two heads.
    constexpr int NP = kHeadsPerLane / 2;
    float2 x2[NP][8];
#pragma unroll
    for (int j = 0; j < NP; ++j)
#pragma unroll
        for (int m = 0; m < 4; ++m) {
            const uint32_t a = word(U.x[2 * j], m), b = word(U.x[2 * j + 1], m);
            x2[j][2 * m] = make_float2(lo_f(a), lo_f(b));
            x2[j][2 * m + 1] = make_float2(hi_f(a), hi_f(b));
        }

    // Partial sum of squares of each of the lane's heads over its 8 columns:
    // one ordered chain per head, rn(acc + rn(x * x)) in column order, two
    // heads per packed operation.
    float ps[16];
#pragma unroll
    for (int j = 0; j < NP; ++j) {
        float2 acc = make_float2(0.0f, 0.0f);
#pragma unroll
        for (int e = 0; e < 8; ++e) acc = addmul2(acc, x2[j][e], x2[j][e]);
        ps[2 * j] = acc.x;
        ps[2 * j + 1] = acc.y;
    }
#pragma unroll
    for (int k = kHeadsPerLane; k < 16; ++k) ps[k] = 0.0f;

    // Recursive-halving fold over the head's LPH lanes: at xor offset 1, 2,
    // .. each lane keeps half of its entries and adds its partner's partial
    // for them.  Per head this is exactly the adjacent-pair tree over the
    // lanes; afterwards lane fl holds the sums of heads NK*brev(fl) + j.
#pragma unroll
    for (int lvl = 0, n = 16; lvl < S::LEVELS; ++lvl, n >>= 1) {
        const int off = 1 << lvl;
        const bool upper = (fl & off) != 0;
#pragma unroll
        for (int i = 0; i < n / 2; ++i) {
            const float send = upper ? ps[i] : ps[i + n / 2];
            const float keep = upper ? ps[i + n / 2] : ps[i];
            ps[i] = __fadd_rn(keep, __shfl_xor_sync(kFull, send, off));
        }
    }
    float my_rstd[S::NK];
#pragma unroll
    for (int j = 0; j < S::NK; ++j)
        my_rstd[j] = defined_rsqrt(__fadd_rn(div_by<HD>(ps[j]), p.eps[U.s_]));

    float2 wd[8], cc[4], sn[4]; // wd[e]: weight of column e, duplicated
#pragma unroll
    for (int m = 0; m < 4; ++m) {
        wd[2 * m] = dup2(lo_f(word(U.w, m)));
        wd[2 * m + 1] = dup2(hi_f(word(U.w, m)));
    }
    const bool first = fl < S::LPH / 2; // neox: the lane holds the first half's columns
    if (NEOX) {
        // columns (2m, 2m+1) of the lane: cos pairs and sin pairs, the sin
        // negated in the first half so both halves add: out = own*c + other*s'
#pragma unroll
        for (int m = 0; m < 4; ++m) {
            const float4 &c4 = U.c[m / 2], &s4 = U.s[m / 2];
            cc[m] = make_float2(f4(c4, 2 * (m % 2)), f4(c4, 2 * (m % 2) + 1));
            const float2 s2 = make_float2(f4(s4, 2 * (m % 2)), f4(s4, 2 * (m % 2) + 1));
            sn[m] = first ? make_float2(-s2.x, -s2.y) : s2;
        }
    } else {
#pragma unroll
        for (int m = 0; m < 4; ++m) {
            cc[m] = dup2(f4(U.c[0], m));
            sn[m] = dup2(f4(U.s[0], m));
        }
    }
    const int lane_base = hs * S::LPH;
    // Rotate the bf16 row nw of head h (this lane's four column pairs) and
    // store it.
    auto rotate_store = [&](const uint32_t (&nw)[4], int h) {
        uint4 out;
        if (NEOX) {
#pragma unroll
            for (int m = 0; m < 4; ++m) {
                const uint32_t other = __shfl_xor_sync(kFull, nw[m], S::LPH / 2);
                const float2 xc = mul2(wide2(nw[m]), cc[m]);  // rn(own * c)
                const float2 ys = mul2(wide2(other), sn[m]);  // rn(other * (-+ s))
                set_word(out, m, pack_bf16(__fadd_rn(xc.x, ys.x), __fadd_rn(xc.y, ys.y)));
            }
        } else {
#pragma unroll
            for (int m = 0; m < 4; ++m) { // pair i = 4fl + m: columns 2i, 2i+1
                const float2 ab = wide2(nw[m]);       // (a, b)
                const float2 pc = mul2(ab, cc[m]);    // (rn(a c), rn(b c))
                const float2 ps2 = mul2(ab, sn[m]);   // (rn(a s), rn(b s))
                set_word(out, m, pack_bf16(__fsub_rn(pc.x, ps2.y), __fadd_rn(ps2.x, pc.y)));
            }
        }
        if (h < p.H) st_stream(dst + h * S::LPH + fl, out);
    };
#pragma unroll
    for (int j = 0; j < NP; ++j) {
        const int k0 = 2 * j, k1 = 2 * j + 1;
        const float r0 = __shfl_sync(kFull, my_rstd[k0 % S::NK], lane_base + brev<S::LEVELS>(k0 / S::NK));
        const float r1 = __shfl_sync(kFull, my_rstd[k1 % S::NK], lane_base + brev<S::LEVELS>(k1 / S::NK));
        if (U.h0 + S::GPS * k0 >= p.H) break; // warp-uniform: no head left in any slot
        const float2 r2 = make_float2(r0, r1);
        // normalised, rounded to bf16: nw0 for head 2j, nw1 for head 2j+1
        uint32_t nw0[4], nw1[4];
#pragma unroll
        for (int m = 0; m < 4; ++m) {
            const float2 te = mul2(mul2(x2[j][2 * m], r2), wd[2 * m]);
            const float2 to = mul2(mul2(x2[j][2 * m + 1], r2), wd[2 * m + 1]);
            nw0[m] = pack_bf16(te.x, to.x);
            nw1[m] = pack_bf16(te.y, to.y);
        }
        rotate_store(nw0, U.h0 + hs + S::GPS * k0);
        if (U.h0 + S::GPS * k1 >= p.H) break;
        rotate_store(nw1, U.h0 + hs + S::GPS * k1);
    }
}

// CTA c takes the tokens c, c + G, c + 2G, ... (measured faster than a
// contiguous block of tokens per CTA: 25.06 against 25.9 us at 256 + 4096
// tokens x 24 heads x 128, and by 0.3 to 1.0 us for the neox and
// head_dim-64 forms); its warp w takes the CTA's units w, w + kQkNW, ...
// and requests each kQkSPC units ahead
// into its own slots (dan_ring.cuh): one bulk copy of the unit's heads,
// plus one of the token's cos/sin row for Q and K.  The four weight
// vectors are staged in shared memory once per CTA.
template <int HD, bool NEOX>
__global__ void __launch_bounds__(32 * kQkNW, 1) qk_norm_rope_kernel(const QkParams p)
{
    using S = QkShape<HD>;
    using Pipe = WarpPipe<kQkSPC>;
    extern __shared__ __align__(128) uint4 smem[];
    uint4 *ring = smem;
    uint4 *s_w = ring + kQkNW * kQkSPC * S::SLOT; // 4 x LPH fragments
    uint64_t *full = reinterpret_cast<uint64_t *>(s_w + 4 * S::LPH);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int hs = lane / S::LPH, fl = lane % S::LPH;
    const int64_t G = gridDim.x;
    const int64_t t0 = blockIdx.x; // the CTA's tokens t0 + G * j
    const int n = (int)((p.T_all - t0 + G - 1) / G * 3 * p.groups);

    const int units = warp < n ? (n - warp + kQkNW - 1) / kQkNW : 0;
    if (lane == 0) // L2 prefetch of the first units: they stream while the previous grid drains
        for (int i = 0; i < kQkPre && i < units; ++i) {
            QkUnit U;
            qk_unit<HD>(U, p, t0, warp + kQkNW * i);
            prefetch_l2(qk_src<HD>(U, p), (unsigned)qk_heads<HD>(U, p) * (unsigned)(HD * 2));
            if (U.kind != 2) prefetch_l2(qk_rope_row<HD>(U, p), HD * 4u);
        }
    if (threadIdx.x == 0) {
        for (int s = 0; s < kQkNW * kQkSPC; ++s) mbar_init(full + s, 1);
        mbar_init_fence();
    }
    grid_dependency_wait(); // no global read above this line (L2 prefetches only)
    allow_dependents();
    if (threadIdx.x < 4 * S::LPH) { // the weights of a stream with no tokens are never read
        const int v = threadIdx.x / S::LPH, s = v >> 1;
        if (s == 0 ? p.T0 > 0 : p.T_all > p.T0)
            s_w[threadIdx.x] = ld_vec((v & 1 ? p.wk[s] : p.wq[s]) + (threadIdx.x % S::LPH));
    }
    __syncthreads(); // barriers initialised, weights staged

    uint4 *slots = ring + warp * kQkSPC * S::SLOT;
    uint64_t *bar = full + warp * kQkSPC;
    auto request = [&](int i) { // lane 0 only
        QkUnit U;
        qk_unit<HD>(U, p, t0, warp + kQkNW * i);
        const unsigned bytes = (unsigned)qk_heads<HD>(U, p) * (unsigned)(HD * 2);
        uint4 *slot = slots + Pipe::slot(i) * S::SLOT;
        uint64_t *b = bar + Pipe::slot(i);
        if (U.kind == 2) {
            mbar_arrive_expect_tx(b, bytes);
            bulk_load(slot, qk_src<HD>(U, p), bytes, b);
        } else {
            mbar_arrive_expect_tx(b, bytes + HD * 4u);
            bulk_load(slot, qk_src<HD>(U, p), bytes, b);
            bulk_load(slot + S::DATA, qk_rope_row<HD>(U, p), HD * 4u, b);
        }
    };
    if (lane == 0)
        for (int i = 0; i < kQkSPC && i < units; ++i) request(i);

    for (int i = 0; i < units; ++i) {
        if (!Pipe::wait(bar, i, p.limit_ns)) {
            Pipe::abort(bar, i, units, p.status, p.limit_ns);
            return;
        }
        QkUnit U;
        qk_unit<HD>(U, p, t0, warp + kQkNW * i);
        qk_take<HD, NEOX>(U, p, slots + Pipe::slot(i) * S::SLOT, s_w, hs, fl);
        slot_reads_done();
        if (lane == 0 && i + kQkSPC < units) request(i + kQkSPC);
        qk_process<HD, NEOX>(U, p, hs, fl);
    }
}

namespace {

template <int HD, bool NEOX>
cudaError_t launch_qk(QkParams p, int64_t heads, cudaStream_t s)
{
    using S = QkShape<HD>;
    p.groups = (int)((heads + S::GROUP - 1) / S::GROUP);
    constexpr int NS = kQkNW * kQkSPC;
    const int smem = NS * S::SLOT * 16 + 4 * S::LPH * 16 + NS * 8;
    auto fn = qk_norm_rope_kernel<HD, NEOX>;
    const cudaError_t e = allow_dynamic_smem(reinterpret_cast<const void *>(fn), smem);
    if (e != cudaSuccess) return e;
    const int grid = (int)(p.T_all < sm_count() ? p.T_all : sm_count());
    return launch_overlapped(fn, grid, 32 * kQkNW, smem, s, p);
}

} // namespace

cudaError_t launch_qk_norm_rope(const QkProblem &q, bool neox, cudaStream_t s)
{
    QkParams p;
    for (int i = 0; i < 2; ++i) {
        p.q[i] = static_cast<const uint4 *>(q.q[i]);
        p.k[i] = static_cast<const uint4 *>(q.k[i]);
        p.v[i] = static_cast<const uint4 *>(q.v[i]);
        p.stride8[i] = q.stride[i] / 8;
        p.wq[i] = static_cast<const uint4 *>(q.wq[i]);
        p.wk[i] = static_cast<const uint4 *>(q.wk[i]);
        p.rope[i] = reinterpret_cast<const float4 *>(q.rope[i]);
        p.eps[i] = q.eps[i];
    }
    p.T0 = q.T[0];
    p.T_all = q.T[0] + q.T[1];
    p.q_out = static_cast<uint4 *>(q.q_out);
    p.k_out = static_cast<uint4 *>(q.k_out);
    p.v_out = static_cast<uint4 *>(q.v_out);
    p.H = (int)q.heads;
    p.groups = 0;
    p.status = device_status();
    p.limit_ns = 1000000000ull;
    if (q.head_dim == 64)
        return neox ? launch_qk<64, true>(p, q.heads, s) : launch_qk<64, false>(p, q.heads, s);
    return neox ? launch_qk<128, true>(p, q.heads, s) : launch_qk<128, false>(p, q.heads, s);
}

} // namespace dan
