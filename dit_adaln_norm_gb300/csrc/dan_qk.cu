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
// Work unit = (token, Q|K|V), one warp each, grid-stride over units.  A
// half-warp covers one head: lane l (0..15) owns the 16-byte fragment of
// columns 8l..8l+7, so each head is one coalesced 256-byte load/store and
// the two halves of a warp take adjacent heads (512 contiguous bytes).  The
// per-token RoPE row and the stream's weight fragment are read once per unit.
// Head RMS: each lane's 8 squares in column order, then the adjacent-pair
// tree over the 16 lanes (xor 1,2,4,8 stays inside a half-warp).
#include "dan_device.cuh"
#include "dan_internal.h"

namespace dan {

struct QkParams {
    const uint4 *q[2], *k[2], *v[2];
    int64_t T0;        // text tokens
    int64_t T_all;     // text + image tokens
    int64_t stride8[2]; // row stride in 16-byte fragments
    const uint4 *wq[2], *wk[2];
    const float4 *rope[2];
    float eps[2];
    uint4 *q_out, *k_out, *v_out;
    int H;
};

constexpr int kQkWarps = 8;
constexpr int kHeadsPerLane = 12; // heads held in registers per half-warp pass

__global__ void __launch_bounds__(kQkWarps * 32) qk_norm_rope_kernel(const QkParams p)
{
    const int lane = threadIdx.x & 31;
    const int half = lane >> 4, fl = lane & 15;
    const int64_t nwarps = (int64_t)gridDim.x * kQkWarps;
    const int64_t units = 3 * p.T_all;

    for (int64_t u = (int64_t)blockIdx.x * kQkWarps + (threadIdx.x >> 5); u < units; u += nwarps) {
        const int64_t tok = u / 3;
        const int kind = (int)(u - 3 * tok); // 0 = Q, 1 = K, 2 = V
        const int s = tok < p.T0 ? 0 : 1;
        const int64_t t = s ? tok - p.T0 : tok;
        const uint4 *src = (kind == 0 ? p.q[s] : kind == 1 ? p.k[s] : p.v[s]) + t * p.stride8[s];
        uint4 *dst = (kind == 0 ? p.q_out : kind == 1 ? p.k_out : p.v_out) + tok * p.H * 16;

        if (kind == 2) { // V: bit copy
            for (int h = half; h < p.H; h += 2) st_stream(dst + h * 16 + fl, ld_stream(src + h * 16 + fl));
            continue;
        }

        const uint4 w = ld_vec((kind == 0 ? p.wq[s] : p.wk[s]) + fl);
        const float4 c4 = ld_vec(p.rope[s] + t * 32 + fl);      // cos of pairs 4fl..4fl+3
        const float4 s4 = ld_vec(p.rope[s] + t * 32 + 16 + fl); // sin of the same pairs
        const float cs[4] = {c4.x, c4.y, c4.z, c4.w};
        const float sn[4] = {s4.x, s4.y, s4.z, s4.w};
        const float eps = p.eps[s];

        for (int h0 = 0; h0 < p.H; h0 += 2 * kHeadsPerLane) {
            uint4 x[kHeadsPerLane];
#pragma unroll
            for (int k = 0; k < kHeadsPerLane; ++k) {
                const int h = h0 + half + 2 * k;
                x[k] = h < p.H ? ld_stream(src + h * 16 + fl) : make_uint4(0, 0, 0, 0);
            }
#pragma unroll
            for (int k = 0; k < kHeadsPerLane; ++k) {
                if (h0 + 2 * k >= p.H) break; // warp-uniform: no head left for either half
                const int h = h0 + half + 2 * k;
                float acc = 0.0f;
#pragma unroll
                for (int e = 0; e < 8; ++e) {
                    const float xv = elem(x[k], e);
                    acc = __fadd_rn(acc, __fmul_rn(xv, xv));
                }
#pragma unroll
                for (int off = 1; off < 16; off <<= 1)
                    acc = __fadd_rn(acc, __shfl_xor_sync(kFull, acc, off));
                const float rstd = defined_rsqrt(__fadd_rn(__fdiv_rn(acc, 128.0f), eps));
                uint4 out;
#pragma unroll
                for (int m = 0; m < 4; ++m) { // pair i = 4fl + m: columns 2i, 2i+1
                    const uint32_t xw = word(x[k], m), ww = word(w, m);
                    const uint32_t n = pack_bf16(__fmul_rn(__fmul_rn(lo_f(xw), rstd), lo_f(ww)),
                                                 __fmul_rn(__fmul_rn(hi_f(xw), rstd), hi_f(ww)));
                    const float a = lo_f(n), b = hi_f(n);
                    set_word(out, m,
                             pack_bf16(__fsub_rn(__fmul_rn(a, cs[m]), __fmul_rn(b, sn[m])),
                                       __fadd_rn(__fmul_rn(a, sn[m]), __fmul_rn(b, cs[m]))));
                }
                if (h < p.H) st_stream(dst + h * 16 + fl, out);
            }
        }
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

    int per_sm = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, qk_norm_rope_kernel, kQkWarps * 32,
                                                      0) != cudaSuccess ||
        per_sm < 1)
        per_sm = 1;
    const int64_t units = 3 * p.T_all;
    const int64_t want = (units + kQkWarps - 1) / kQkWarps;
    const int64_t cap = (int64_t)sm_count() * per_sm;
    const int grid = (int)(want < cap ? want : cap);
    qk_norm_rope_kernel<<<grid, kQkWarps * 32, 0, s>>>(p);
    return cudaGetLastError();
}

} // namespace dan
