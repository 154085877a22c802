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

constexpr int kQkNC = 8;  // consumer warps per CTA
constexpr int kQkSPC = 2; // ring slots per consumer
constexpr int kHeadsPerLane = 12;           // heads a half-warp lane holds per unit
constexpr int kGroup = 2 * kHeadsPerLane;   // heads per unit

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
    const int per_tok = 3 * p.groups;
    U.tok = t0 + k / per_tok;
    const int rem = k % per_tok;
    U.kind = rem / p.groups;
    U.h0 = (rem % p.groups) * kGroup;
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

// Copy the unit's heads from its ring slot into registers, and read the
// stream's weight fragment and the token's cos/sin for Q and K.
__device__ __forceinline__ void qk_take(QkUnit &U, const QkParams &p, const uint4 *slot, int half,
                                        int fl)
{
    const int nh = qk_heads(U, p);
#pragma unroll
    for (int k = 0; k < kHeadsPerLane; ++k) {
        const int hh = half + 2 * k;
        U.x[k] = hh < nh ? slot[hh * 16 + fl] : make_uint4(0, 0, 0, 0);
    }
    if (U.kind != 2) {
        const int64_t t = U.s ? U.tok - p.T0 : U.tok;
        U.w = ld_vec((U.kind == 0 ? p.wq[U.s] : p.wk[U.s]) + fl);
        U.c4 = ld_vec(p.rope[U.s] + t * 32 + fl);      // cos of pairs 4fl..4fl+3
        U.s4 = ld_vec(p.rope[U.s] + t * 32 + 16 + fl); // sin of the same pairs
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

    // Partial sum of squares of each of the lane's heads over its 8 columns
    // (one ordered chain per head; heads k, k+1 share packed multiplies).
    float ps[16];
#pragma unroll
    for (int k = 0; k < kHeadsPerLane; k += 2) {
        float2 acc = make_float2(0.0f, 0.0f);
#pragma unroll
        for (int e = 0; e < 8; ++e) {
            const float2 x2 = make_float2(elem(U.x[k], e), elem(U.x[k + 1], e));
            acc = addmul2(acc, x2, x2);
        }
        ps[k] = acc.x;
        ps[k + 1] = acc.y;
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

    const float cs[4] = {U.c4.x, U.c4.y, U.c4.z, U.c4.w};
    const float sn[4] = {U.s4.x, U.s4.y, U.s4.z, U.s4.w};
    float2 w2[4];
#pragma unroll
    for (int m = 0; m < 4; ++m) w2[m] = wide2(word(U.w, m));
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
            const float2 t2 = mul2(mul2(wide2(word(U.x[k], m)), r2), w2[m]);
            const uint32_t n = pack_bf16(t2.x, t2.y);
            const float a = lo_f(n), b = hi_f(n);
            set_word(out, m,
                     pack_bf16(__fsub_rn(__fmul_rn(a, cs[m]), __fmul_rn(b, sn[m])),
                               __fadd_rn(__fmul_rn(a, sn[m]), __fmul_rn(b, cs[m]))));
        }
        if (h < p.H) st_stream(dst + h * 16 + fl, out);
    }
}

// CTA c takes the contiguous tokens [c*T/G, (c+1)*T/G) and streams their
// units through a ring of 6 KB slots (dan_ring.cuh): warp 0 lane 0 issues
// one bulk copy per unit, warps 1..kQkNC consume.
__global__ void __launch_bounds__(32 * (kQkNC + 1), 1) qk_norm_rope_kernel(const QkParams p)
{
    using R = RingSchedule<kQkNC, kQkSPC>;
    constexpr int kSlot = kGroup * 16; // uint4 per slot
    extern __shared__ __align__(128) uint4 smem[];
    uint4 *ring = smem;
    uint64_t *full = reinterpret_cast<uint64_t *>(ring + R::S * kSlot);
    uint64_t *empty = full + R::S;

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int half = (lane >> 4) & 1, fl = lane & 15;
    const int64_t G = gridDim.x;
    const int64_t t0 = (int64_t)blockIdx.x * p.T_all / G;
    const int64_t t1 = (int64_t)(blockIdx.x + 1) * p.T_all / G;
    const int n = (int)((t1 - t0) * 3 * p.groups);

    if (threadIdx.x == 0) {
        for (int s = 0; s < R::S; ++s) {
            mbar_init(full + s, 1);
            mbar_init(empty + s, 1);
        }
        mbar_init_fence();
    }
    __syncthreads();

    if (warp == 0) {
        if (lane == 0)
            ring_produce<kQkNC, kQkSPC>(n, full, empty, p.status, p.limit_ns, [&](int k, int s) {
                QkUnit U;
                qk_unit(U, p, t0, k);
                const unsigned bytes = (unsigned)qk_heads(U, p) * 256u;
                mbar_arrive_expect_tx(full + s, bytes);
                bulk_load(ring + s * kSlot, qk_src(U, p), bytes, full + s);
            });
        return;
    }

    const int c = warp - 1;
    for (int i = 0;; ++i) {
        const int k = c + i * kQkNC;
        if (k >= n) break;
        const int s = R::slot(c, i);
        if (!mbar_wait(full + s, R::phase(i), p.limit_ns)) {
            set_status(p.status, kStatusWaitFull);
            return;
        }
        QkUnit U;
        qk_unit(U, p, t0, k);
        qk_take(U, p, ring + s * kSlot, half, fl);
        ring_release(empty + s, lane);
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

    constexpr int S = kQkNC * kQkSPC;
    const int smem = S * kGroup * 256 + 2 * S * 8;
    static bool configured = false; // dynamic shared memory above 48 KB (once)
    if (!configured) {
        const cudaError_t e = cudaFuncSetAttribute(
            qk_norm_rope_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
        if (e != cudaSuccess) return e;
        configured = true;
    }
    const int grid = (int)(p.T_all < sm_count() ? p.T_all : sm_count());
    qk_norm_rope_kernel<<<grid, 32 * (kQkNC + 1), smem, s>>>(p);
    return cudaGetLastError();
}

} // namespace dan
