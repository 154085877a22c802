// dan_device.cuh -- device helpers shared by the row kernels and the QK
// epilogue: bf16 <-> fp32 on packed words, 16-byte streaming global access,
// and the defined reciprocal square root.
//
// Every fp32 operation in the kernels goes through the __f*_rn intrinsics
// (one IEEE binary32 operation, round to nearest even, never contracted into
// an FMA); the library is also compiled with -fmad=false.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp8.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace dan {

constexpr unsigned kFull = 0xFFFFFFFFu;

// A 32-bit word holds two bf16 elements: the lower column in the low half.
__device__ __forceinline__ float lo_f(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float hi_f(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }

// Round two fp32 values to bf16 (nearest even) and pack them, a in the low half.
__device__ __forceinline__ uint32_t pack_bf16(float a, float b)
{
    __nv_bfloat162 v = __floats2bfloat162_rn(a, b);
    return *reinterpret_cast<uint32_t *>(&v);
}

// Element e (0..7) of a 16-byte fragment of eight bf16 values, as fp32.
__device__ __forceinline__ float elem(const uint4 &f, int e)
{
    uint32_t w = (e < 2) ? f.x : (e < 4) ? f.y : (e < 6) ? f.z : f.w;
    return (e & 1) ? hi_f(w) : lo_f(w);
}

__device__ __forceinline__ uint32_t word(const uint4 &f, int i)
{
    return i == 0 ? f.x : i == 1 ? f.y : i == 2 ? f.z : f.w;
}

__device__ __forceinline__ void set_word(uint4 &f, int i, uint32_t w)
{
    if (i == 0) f.x = w;
    else if (i == 1) f.y = w;
    else if (i == 2) f.z = w;
    else f.w = w;
}

// Streaming 16-byte global load: coherent path, no L1 allocation (each row
// is read once; in-place calls write it afterwards from the same warp).
__device__ __forceinline__ uint4 ld_stream(const uint4 *p)
{
    uint4 v;
    asm volatile("ld.global.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "l"(p));
    return v;
}

// Streaming 16-byte global store (written once, not re-read by the kernel).
__device__ __forceinline__ void st_stream(uint4 *p, const uint4 &v)
{
    asm volatile("st.global.L1::no_allocate.v4.u32 [%0], {%1,%2,%3,%4};" ::"l"(p), "r"(v.x),
                 "r"(v.y), "r"(v.z), "r"(v.w)
                 : "memory");
}

// Streaming 8-byte global store.
__device__ __forceinline__ void st_stream8(uint2 *p, const uint2 &v)
{
    asm volatile("st.global.L1::no_allocate.v2.u32 [%0], {%1,%2};" ::"l"(p), "r"(v.x), "r"(v.y)
                 : "memory");
}

// Two fp32 values to FP8 E4M3 codes (round to nearest even, saturated to the
// largest finite value), v.x in the low byte.
__device__ __forceinline__ uint32_t fp8x2_e4m3(float2 v)
{
    return (uint32_t)__nv_cvt_float2_to_fp8x2(v, __NV_SATFINITE, __NV_E4M3);
}

// Asynchronous 16-byte global -> shared copy (bypassing L1), and the wait
// for all of this thread's outstanding copies (a hardware wait on the
// thread's own copy group, like a load dependency; no polling loop).
__device__ __forceinline__ void cp_async16(void *smem_dst, const void *gmem_src)
{
    const unsigned d = (unsigned)__cvta_generic_to_shared(smem_dst);
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(d), "l"(gmem_src) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
__device__ __forceinline__ void cp_async_wait_all() { asm volatile("cp.async.wait_group 0;" ::: "memory"); }
// Wait until at most N of this thread's committed groups are still in flight.
template <int N>
__device__ __forceinline__ void cp_async_wait() { asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory"); }

// Read-only 16-byte load of a small broadcast vector (kept in L1/L2).
__device__ __forceinline__ uint4 ld_vec(const uint4 *p) { return __ldg(p); }
__device__ __forceinline__ float4 ld_vec(const float4 *p) { return __ldg(p); }

// rn(x / D) for a divisor D known at compile time.  For a power of two it
// is the multiply by the exact reciprocal 2^-k: both give the exact
// quotient rounded once, so the bits are those of the IEEE division.
template <int D>
__device__ __forceinline__ float div_by(float x)
{
    if constexpr ((D & (D - 1)) == 0) return __fmul_rn(x, 1.0f / (float)D);
    else return __fdiv_rn(x, (float)D);
}

// The defined reciprocal square root: rn(1 / rn(sqrt(v))), two IEEE ops.
__device__ __forceinline__ float defined_rsqrt(float v)
{
    return __fdiv_rn(1.0f, __fsqrt_rn(v));
}

// ------------------------------------------------ packed fp32x2 (sm_100+)
// Each lane of a packed operation is one IEEE binary32 operation rounded to
// nearest even, exactly as the scalar __f*_rn forms.  They are written as
// PTX with an explicit .rn qualifier: such operations are never contracted
// into an FMA (a fused multiply-add would round once where the method
// rounds twice, e.g. in the Welford update mean + d * rn(1/n)).

__device__ __forceinline__ uint64_t pk2(float2 a)
{
    uint64_t u;
    asm("mov.b64 %0, {%1,%2};" : "=l"(u) : "f"(a.x), "f"(a.y));
    return u;
}
__device__ __forceinline__ float2 upk2(uint64_t u)
{
    float2 o;
    asm("mov.b64 {%0,%1}, %2;" : "=f"(o.x), "=f"(o.y) : "l"(u));
    return o;
}
__device__ __forceinline__ float2 add2(float2 a, float2 b)
{
    uint64_t r;
    asm("add.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(pk2(a)), "l"(pk2(b)));
    return upk2(r);
}
__device__ __forceinline__ float2 sub2(float2 a, float2 b)
{
    uint64_t r;
    asm("sub.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(pk2(a)), "l"(pk2(b)));
    return upk2(r);
}
__device__ __forceinline__ float2 mul2(float2 a, float2 b)
{
    uint64_t r;
    asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(pk2(a)), "l"(pk2(b)));
    return upk2(r);
}
// acc + rn(a * b) per lane, the sum rounded separately, for accumulators
// that are never -0.  ptxas (CUDA 13.0) was measured to contract a packed
// mul.rn.f32x2 feeding a packed add.rn.f32x2 into one fused multiply-add
// inside unrolled chains, despite the explicit .rn and --fmad=false (and a
// fused multiply-add with a -0 addend, the exact identity of a multiply,
// the same way).  So the product is formed as fma(a, b, +0): that equals
// rn(a * b) except that a -0 product becomes +0, and acc + (+0) equals
// acc + (-0) unless acc is -0.  The accumulators this serves (sums of
// squares, Welford means and m2, and their combines) start at +0 and can
// never become -0, because a round-to-nearest sum is -0 only when both
// addends are -0.  Two instructions instead of a multiply and two adds.
__device__ __forceinline__ float2 addmul2(float2 acc, float2 a, float2 b)
{
    const uint64_t pos_zero = 0; // (+0, +0)
    uint64_t t, r;
    asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(t) : "l"(pk2(a)), "l"(pk2(b)), "l"(pos_zero));
    asm("add.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(pk2(acc)), "l"(t));
    return upk2(r);
}
__device__ __forceinline__ float2 dup2(float a) { return make_float2(a, a); }
// Both elements of a bf16 word as a float2 (low column first).
__device__ __forceinline__ float2 wide2(uint32_t w) { return make_float2(lo_f(w), hi_f(w)); }

// ------------------------------------------------------- bf16x2 arithmetic
// For bf16 operands these equal the fp32-then-round chain bit for bit:
//  * a*b: the exact product of two bf16 values has at most 16 significant
//    bits and, when its magnitude is at least 2^-134, no bit below 2^-149,
//    so rn32(a*b) is exact; below 2^-134 both roundings give a signed zero.
//    Hence bf16(rn32(a*b)) == bf16_rn(a*b).
//  * a+b: when the exponents differ by at most 15 the exact sum fits in 24
//    bits (rn32 exact); otherwise the smaller term is below 2^-15 of the
//    larger, far from any bf16 rounding midpoint, and both give the same.
__device__ __forceinline__ uint32_t hmul2(uint32_t a, uint32_t b)
{
    uint32_t r;
    asm("mul.rn.bf16x2 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(b));
    return r;
}
__device__ __forceinline__ uint32_t hadd2(uint32_t a, uint32_t b)
{
    uint32_t r;
    asm("add.rn.bf16x2 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(b));
    return r;
}

// o = bf16(rn(1 + scale)) for the eight elements of a scale fragment.
__device__ __forceinline__ uint4 one_plus_fragment(const uint4 &sc)
{
    uint4 o;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        uint32_t w = word(sc, i);
        set_word(o, i, pack_bf16(__fadd_rn(1.0f, lo_f(w)), __fadd_rn(1.0f, hi_f(w))));
    }
    return o;
}

// The modulate chain on one word (two elements) of normalised values n
// (already bf16): y = bf16(rn(bf16(rn(n * o)) + shift)), as bf16x2 ops.
__device__ __forceinline__ uint32_t modulate_word(uint32_t n, uint32_t o, uint32_t sh)
{
    return hadd2(hmul2(n, o), sh);
}

// Gated residual on one word: r' = bf16(rn(r + bf16(rn(gate * h)))).
__device__ __forceinline__ uint32_t gated_word(uint32_t r, uint32_t g, uint32_t h)
{
    return hadd2(r, hmul2(g, h));
}

} // namespace dan
