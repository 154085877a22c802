// dan_qk.cu -- QK-RMSNorm + interleaved RoPE + V copy epilogue for sm_103a.
//
// "PR #37123 report" (Qwen-Image FP8 QKV projection and Blackwell
// epilogue), implementation section 3: one kernel walks the Q/K/V work of
// the text and image token streams, normalises every 128-wide head of Q and
// K with that stream's RMSNorm weight, rotates interleaved pairs with the
// stream's fp32 cos/sin row, copies V, and writes joint [text, image]
// buffers; inputs are zero-copy row-strided views of the packed QKV GEMM
// output (section 4).
//
// Work unit = (token, Q|K|V, group of up to 24 heads): one bulk copy into
// a shared-memory ring slot, processed by one consumer warp (see
// dan_ring.cuh for the ring).  A half-warp covers one head: lane l (0..15) owns the 16-byte fragment of
// columns 8l..8l+7, so each head is one coalesced 256-byte load/store and
// the two halves of a warp take adjacent heads (512 contiguous bytes).  The
// per-token RoPE row and the stream's weight fragment are read once per unit.
// Head RMS: each lane's 8 squares in column order, then the adjacent-pair
// tree over the 16 lanes (xor 1,2,4,8 stays inside a half-warp), done as a
// recursive-halving fold so that each lane ends with one head's sum.
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
    int groups; // head groups of kGroup heads per (token, kind)
    unsigned *status;
    unsigned long long limit_ns;
};

constexpr int kQkNW = 8;  // warps per CTA (measured best among 4..16)
constexpr int kQkSPC = 1; // slots per warp
constexpr int kHeadsPerLane = 12;         // heads a half-warp lane holds per unit
constexpr int kGroup = 2 * kHeadsPerLane; // heads per unit
// A ring slot holds one unit's heads (16 fragments each) and, for Q and K,
// the token's cos/sin row (128 fp32 = 32 fragments) behind them.
constexpr int kSlotRope = kGroup * 16;
constexpr int kSlot = kSlotRope + 32;

// One unit of work = (token, Q|K|V, group of up to kGroup heads), as
// loaded registers: the head fragments plus, for Q and K, the weight
// fragment and the token's cos/sin for this lane's four pairs.
struct QkUnit {
    uint4 x[kHeadsPerLane];
    uint4 w;
    float4 c4, s4;
    int64_t tok;
    int kind, h0, s;
};

// Unit k of a CTA whose tokens start at t0: token t0 + k / (3 * groups),
// then Q, K, V, each split in head groups.
__device__ __forceinline__ void qk_unit(QkUnit &U, const QkParams &p, int64_t t0, int k)
{
    if (p.groups == 1) { // up to kGroup heads: one unit per (token, kind); k / 3 by a constant
        const unsigned uk = (unsigned)k;
        U.tok = t0 + uk / 3u;
        U.kind = (int)(uk % 3u);
        U.h0 = 0;
    } else {
        const int per_tok = 3 * p.groups;
        U.tok = t0 + k / per_tok;
        const int rem = k % per_tok;
        U.kind = rem / p.groups;
        U.h0 = (rem % p.groups) * kGroup;
    }
    U.s = U.tok < p.T0 ? 0 : 1;
}

__device__ __forceinline__ const uint4 *qk_src(const QkUnit &U, const QkParams &p)
{
    const int64_t t = U.s ? U.tok - p.T0 : U.tok;
    return (U.kind == 0 ? p.q[U.s] : U.kind == 1 ? p.k[U.s] : p.v[U.s]) + t * p.stride8[U.s] +
           U.h0 * 16;
}

__device__ __forceinline__ int qk_heads(const QkUnit &U, const QkParams &p)
{
    return p.H - U.h0 < kGroup ? p.H - U.h0 : kGroup;
}

__device__ __forceinline__ const float4 *qk_rope_row(const QkUnit &U, const QkParams &p)
{
    const int64_t t = U.s ? U.tok - p.T0 : U.tok;
    return p.rope[U.s] + t * 32;
}

// Copy the unit's heads from its ring slot into registers, with, for Q and
// K, the stream's weight fragment (staged in s_w: wq_txt, wk_txt, wq_img,
// wk_img) and the token's cos/sin for this lane's four pairs (in the slot).
__device__ __forceinline__ void qk_take(QkUnit &U, const QkParams &p, const uint4 *slot,
                                        const uint4 *s_w, int half, int fl)
{
    const int nh = qk_heads(U, p);
#pragma unroll
    for (int k = 0; k < kHeadsPerLane; ++k) {
        const int hh = half + 2 * k;
        U.x[k] = hh < nh ? slot[hh * 16 + fl] : make_uint4(0, 0, 0, 0);
    }
    if (U.kind != 2) {
        U.w = s_w[(2 * U.s + U.kind) * 16 + fl];
        const float4 *rope = reinterpret_cast<const float4 *>(slot + kSlotRope);
        U.c4 = rope[fl];      // cos of pairs 4fl..4fl+3
        U.s4 = rope[16 + fl]; // sin of the same pairs
    }
}

// Reverse the 4 low bits: after the halving fold, lane l holds head brev4(l).
__device__ __forceinline__ int brev4(int l)
{
    return ((l & 1) << 3) | ((l & 2) << 1) | ((l & 4) >> 1) | ((l & 8) >> 3);
}

__device__ __forceinline__ void qk_process(const QkUnit &U, const QkParams &p, int half, int fl)
{
    uint4 *dst = (U.kind == 0 ? p.q_out : U.kind == 1 ? p.k_out : p.v_out) + U.tok * p.H * 16;
    if (U.kind == 2) { // V: bit copy
#pragma unroll
        for (int k = 0; k < kHeadsPerLane; ++k) {
            const int h = U.h0 + half + 2 * k;
            if (h < p.H) st_stream(dst + h * 16 + fl, U.x[k]);
        }
        return;
    }

    // The lane's columns widened to fp32 once; packed operations take the
    // two columns of one rotation pair (2i, 2i+1) throughout.
    float x[kHeadsPerLane][8];
#pragma unroll
    for (int k = 0; k < kHeadsPerLane; ++k)
#pragma unroll
        for (int m = 0; m < 4; ++m) {
            x[k][2 * m] = lo_f(word(U.x[k], m));
            x[k][2 * m + 1] = hi_f(word(U.x[k], m));
        }

    // Partial sum of squares of each of the lane's heads over its 8 columns:
    // one ordered chain per head (two products per packed multiply, added
    // in column order).
    float ps[16];
#pragma unroll
    for (int k = 0; k < kHeadsPerLane; ++k) {
        float acc = 0.0f;
#pragma unroll
        for (int e = 0; e < 8; e += 2) {
            const float2 x2 = make_float2(x[k][e], x[k][e + 1]);
            const float2 sq = mul2(x2, x2);
            acc = __fadd_rn(acc, sq.x);
            acc = __fadd_rn(acc, sq.y);
        }
        ps[k] = acc;
    }
#pragma unroll
    for (int k = kHeadsPerLane; k < 16; ++k) ps[k] = 0.0f;

    // Recursive-halving fold over the 16 lanes of the half-warp: at xor
    // offset 1, 2, 4, 8 each lane keeps half of its heads and adds its
    // partner's partial for them.  Per head this is exactly the adjacent-pair
    // tree over the 16 lanes; afterwards lane fl holds the sum of head
    // brev4(fl), so each lane computes one reciprocal square root.
#pragma unroll
    for (int lvl = 0, n = 16; lvl < 4; ++lvl, n >>= 1) {
        const int off = 1 << lvl;
        const bool upper = (fl & off) != 0;
#pragma unroll
        for (int i = 0; i < n / 2; ++i) {
            const float send = upper ? ps[i] : ps[i + n / 2];
            const float keep = upper ? ps[i + n / 2] : ps[i];
            ps[i] = __fadd_rn(keep, __shfl_xor_sync(kFull, send, off));
        }
    }
    const float my_rstd = defined_rsqrt(__fadd_rn(__fdiv_rn(ps[0], 128.0f), p.eps[U.s]));

    // cos and sin of the lane's four pairs, each duplicated for a packed
    // multiply of both members (a, b) of a pair.
    const float cs[4] = {U.c4.x, U.c4.y, U.c4.z, U.c4.w};
    const float sn[4] = {U.s4.x, U.s4.y, U.s4.z, U.s4.w};
    float2 cc[4], ss[4], w2[4];
#pragma unroll
    for (int m = 0; m < 4; ++m) {
        cc[m] = dup2(cs[m]);
        ss[m] = dup2(sn[m]);
        w2[m] = wide2(word(U.w, m));
    }
    const int lane_base = half << 4;
#pragma unroll
    for (int k = 0; k < kHeadsPerLane; ++k) {
        const float rstd = __shfl_sync(kFull, my_rstd, lane_base + brev4(k));
        if (U.h0 + 2 * k >= p.H) break; // warp-uniform: no head left for either half
        const int h = U.h0 + half + 2 * k;
        const float2 r2 = dup2(rstd);
        uint4 out;
#pragma unroll
        for (int m = 0; m < 4; ++m) { // pair i = 4fl + m: columns 2i, 2i+1
            const float2 t2 = mul2(mul2(make_float2(x[k][2 * m], x[k][2 * m + 1]), r2), w2[m]);
            const float2 ab = wide2(pack_bf16(t2.x, t2.y)); // (a, b) rounded to bf16
            const float2 pc = mul2(ab, cc[m]);              // (rn(a c), rn(b c))
            const float2 ps2 = mul2(ab, ss[m]);             // (rn(a s), rn(b s))
            set_word(out, m, pack_bf16(__fsub_rn(pc.x, ps2.y), __fadd_rn(ps2.x, pc.y)));
        }
        if (h < p.H) st_stream(dst + h * 16 + fl, out);
    }
}

// CTA c takes the contiguous tokens [c*T/G, (c+1)*T/G); its warp w takes
// the CTA's units w, w + kQkNW, ... and requests each kQkSPC units ahead
// into its own 6.5 KB slots (dan_ring.cuh): one bulk copy of the unit's
// heads, plus one of the token's cos/sin row for Q and K.  The four
// 256-byte weight vectors are staged in shared memory once per CTA.
__global__ void __launch_bounds__(32 * kQkNW, 1) qk_norm_rope_kernel(const QkParams p)
{
    using Pipe = WarpPipe<kQkSPC>;
    extern __shared__ __align__(128) uint4 smem[];
    uint4 *ring = smem;
    uint4 *s_w = ring + kQkNW * kQkSPC * kSlot; // 4 x 16 fragments
    uint64_t *full = reinterpret_cast<uint64_t *>(s_w + 64);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int half = (lane >> 4) & 1, fl = lane & 15;
    const int64_t G = gridDim.x;
    const int64_t t0 = (int64_t)blockIdx.x * p.T_all / G;
    const int64_t t1 = (int64_t)(blockIdx.x + 1) * p.T_all / G;
    const int n = (int)((t1 - t0) * 3 * p.groups);

    if (threadIdx.x == 0) {
        for (int s = 0; s < kQkNW * kQkSPC; ++s) mbar_init(full + s, 1);
        mbar_init_fence();
    }
    grid_dependency_wait(); // no global access above this line
    allow_dependents();
    if (threadIdx.x < 64) { // the weights of a stream with no tokens are never read
        const int v = threadIdx.x >> 4, s = v >> 1;
        if (s == 0 ? p.T0 > 0 : p.T_all > p.T0)
            s_w[threadIdx.x] = ld_vec((v & 1 ? p.wk[s] : p.wq[s]) + (threadIdx.x & 15));
    }
    __syncthreads(); // barriers initialised, weights staged

    uint4 *slots = ring + warp * kQkSPC * kSlot;
    uint64_t *bar = full + warp * kQkSPC;
    const int units = warp < n ? (n - warp + kQkNW - 1) / kQkNW : 0;
    auto request = [&](int i) { // lane 0 only
        QkUnit U;
        qk_unit(U, p, t0, warp + kQkNW * i);
        const unsigned bytes = (unsigned)qk_heads(U, p) * 256u;
        uint4 *slot = slots + Pipe::slot(i) * kSlot;
        uint64_t *b = bar + Pipe::slot(i);
        if (U.kind == 2) {
            mbar_arrive_expect_tx(b, bytes);
            bulk_load(slot, qk_src(U, p), bytes, b);
        } else {
            mbar_arrive_expect_tx(b, bytes + 512u);
            bulk_load(slot, qk_src(U, p), bytes, b);
            bulk_load(slot + kSlotRope, qk_rope_row(U, p), 512u, b);
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
        qk_unit(U, p, t0, warp + kQkNW * i);
        qk_take(U, p, slots + Pipe::slot(i) * kSlot, s_w, half, fl);
        slot_reads_done();
        if (lane == 0 && i + kQkSPC < units) request(i + kQkSPC);
        qk_process(U, p, half, fl);
    }
}

cudaError_t launch_qk_norm_rope_epilogue(const QkProblem &q, cudaStream_t s)
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
    p.groups = (int)((q.heads + kGroup - 1) / kGroup);
    p.status = device_status();
    p.limit_ns = 1000000000ull;

    constexpr int S = kQkNW * kQkSPC;
    const int smem = S * kSlot * 16 + 64 * 16 + S * 8;
    const cudaError_t e = allow_dynamic_smem(reinterpret_cast<const void *>(qk_norm_rope_kernel), smem);
    if (e != cudaSuccess) return e;
    const int grid = (int)(p.T_all < sm_count() ? p.T_all : sm_count());
    return launch_overlapped(qk_norm_rope_kernel, grid, 32 * kQkNW, smem, s, p);
}

} // namespace dan
