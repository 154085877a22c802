// dan_abi.cu -- the extern "C" boundary: argument validation and launches.
//
// The page's predicate + kernel protocol ("SGLang diffusion fused-op package
// guide", section on entry-point protocol: an unsupported input is an error,
// never a silent fallback) becomes status codes here: every dan_can_use_*
// runs exactly the validation of its entry point and launches nothing.
#include "../../include/dan.h"
#include "dan_internal.h"

#include <cmath>
#include <cstdint>
#include <map>
#include <mutex>
#include <utility>

namespace {

constexpr int64_t kMaxElems = int64_t(1) << 40; // generous bound that keeps byte math in int64

bool al16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

struct Span {
    uintptr_t lo = 0, hi = 0; // [lo, hi); empty when lo == hi
    bool empty() const { return lo == hi; }
};

Span span(const void *p, int64_t bytes)
{
    Span s;
    s.lo = reinterpret_cast<uintptr_t>(p);
    s.hi = s.lo + static_cast<uintptr_t>(bytes);
    return s;
}

bool overlaps(const Span &a, const Span &b)
{
    return !a.empty() && !b.empty() && a.lo < b.hi && b.lo < a.hi;
}

bool eps_ok(float eps) { return std::isfinite(eps) && eps >= 0.0f; }

// Bytes spanned by a [B, D] vector view with batch stride vs.
int64_t vec_bytes(int64_t B, int64_t D, int64_t vs) { return ((B - 1) * vs + D) * 2; }

// Shared checks of the three row operations.  `ins` are inputs (nullptr
// entries skipped), `outs` outputs; `same_ok[i]` names the input that output
// i may equal exactly (in-place), or -1.
int check_rows(int64_t B, int64_t T, int64_t D, float eps, int64_t vs, bool d_ok)
{
    if (B < 0 || T < 0 || D < 0) return DAN_EINVAL;
    if (!d_ok) return DAN_EUNSUPPORTED;
    if (!eps_ok(eps)) return DAN_EINVAL;
    if (B > 0 && T > kMaxElems / B) return DAN_EINVAL;
    if (B * T > kMaxElems / D) return DAN_EINVAL;
    if (B * T == 0) return DAN_OK;
    if (vs < D || vs > kMaxElems || (B - 1) > kMaxElems / vs) return DAN_EINVAL;
    if (vs % 8) return DAN_EALIGN;
    return DAN_OK;
}

bool rms_d_ok(int64_t D) { return D == 2048 || D == 4096 || D == 6144 || D == 8192; }
bool ln_d_ok(int64_t D) { return D >= 8 && D <= 8192 && D % 8 == 0; }

struct Buf {
    const void *p;
    Span s;
};

// Validate pointers of a row call: every listed pointer non-null and
// aligned; outputs disjoint from inputs and each other except exact
// in-place pairs (out index, in index).
int check_buffers(const Buf *ins, int nin, const Buf *outs, int nout, const int (*inplace)[2],
                  int ninplace)
{
    for (int i = 0; i < nin; ++i) {
        if (!ins[i].p) return DAN_EINVAL;
    }
    for (int i = 0; i < nout; ++i) {
        if (!outs[i].p) return DAN_EINVAL;
    }
    for (int i = 0; i < nin; ++i)
        if (!al16(ins[i].p)) return DAN_EALIGN;
    for (int i = 0; i < nout; ++i)
        if (!al16(outs[i].p)) return DAN_EALIGN;
    for (int o = 0; o < nout; ++o) {
        for (int i = 0; i < nin; ++i) {
            bool allowed = false;
            for (int k = 0; k < ninplace; ++k)
                if (inplace[k][0] == o && inplace[k][1] == i && outs[o].p == ins[i].p &&
                    outs[o].s.hi == ins[i].s.hi)
                    allowed = true;
            if (!allowed && overlaps(outs[o].s, ins[i].s)) return DAN_EALIAS;
        }
        for (int o2 = o + 1; o2 < nout; ++o2)
            if (overlaps(outs[o].s, outs[o2].s)) return DAN_EALIAS;
    }
    return DAN_OK;
}

int validate_rms(const dan_bf16 *x, const dan_bf16 *weight, const dan_bf16 *scale,
                 const dan_bf16 *shift, int64_t vs, const dan_bf16 *y, int64_t B, int64_t T,
                 int64_t D, float eps, bool *empty)
{
    int st = check_rows(B, T, D, eps, vs, rms_d_ok(D));
    *empty = (st == DAN_OK && B * T == 0);
    if (st != DAN_OK || *empty) return st;
    const int64_t rows = B * T * D * 2;
    Buf ins[4] = {{x, span(x, rows)}, {scale, span(scale, vec_bytes(B, D, vs))},
                  {shift, span(shift, vec_bytes(B, D, vs))}, {weight, span(weight, D * 2)}};
    Buf outs[1] = {{y, span(y, rows)}};
    const int inplace[1][2] = {{0, 0}};
    return check_buffers(ins, weight ? 4 : 3, outs, 1, inplace, 1);
}

int validate_gated(const dan_bf16 *r, const dan_bf16 *h, const dan_bf16 *gate,
                   const dan_bf16 *weight, const dan_bf16 *scale, const dan_bf16 *shift,
                   int64_t vs, const dan_bf16 *r_out, const dan_bf16 *y, int64_t B, int64_t T,
                   int64_t D, float eps, bool *empty)
{
    int st = check_rows(B, T, D, eps, vs, rms_d_ok(D));
    *empty = (st == DAN_OK && B * T == 0);
    if (st != DAN_OK || *empty) return st;
    const int64_t rows = B * T * D * 2, vb = vec_bytes(B, D, vs);
    Buf ins[6] = {{r, span(r, rows)},         {h, span(h, rows)},
                  {gate, span(gate, vb)},     {scale, span(scale, vb)},
                  {shift, span(shift, vb)},   {weight, span(weight, D * 2)}};
    Buf outs[2] = {{r_out, span(r_out, rows)}, {y, span(y, rows)}};
    const int inplace[1][2] = {{0, 0}}; // r_out == r
    return check_buffers(ins, weight ? 6 : 5, outs, 2, inplace, 1);
}

int validate_ln(const dan_bf16 *x, const dan_bf16 *scale, const dan_bf16 *shift, int64_t vs,
                const dan_bf16 *y, int64_t B, int64_t T, int64_t D, float eps, bool *empty)
{
    int st = check_rows(B, T, D, eps, vs, ln_d_ok(D));
    *empty = (st == DAN_OK && B * T == 0);
    if (st != DAN_OK || *empty) return st;
    const int64_t rows = B * T * D * 2;
    Buf ins[3] = {{x, span(x, rows)}, {scale, span(scale, vec_bytes(B, D, vs))},
                  {shift, span(shift, vec_bytes(B, D, vs))}};
    Buf outs[1] = {{y, span(y, rows)}};
    const int inplace[1][2] = {{0, 0}};
    return check_buffers(ins, 3, outs, 1, inplace, 1);
}

int validate_gated_ln(const dan_bf16 *r, const dan_bf16 *h, const dan_bf16 *gate,
                      const dan_bf16 *scale, const dan_bf16 *shift, int64_t vs,
                      const dan_bf16 *r_out, const dan_bf16 *y, int64_t B, int64_t T, int64_t D,
                      float eps, bool *empty)
{
    int st = check_rows(B, T, D, eps, vs, ln_d_ok(D));
    *empty = (st == DAN_OK && B * T == 0);
    if (st != DAN_OK || *empty) return st;
    const int64_t rows = B * T * D * 2, vb = vec_bytes(B, D, vs);
    Buf ins[5] = {{r, span(r, rows)},     {h, span(h, rows)},       {gate, span(gate, vb)},
                  {scale, span(scale, vb)}, {shift, span(shift, vb)}};
    Buf outs[2] = {{r_out, span(r_out, rows)}, {y, span(y, rows)}};
    const int inplace[1][2] = {{0, 0}}; // r_out == r
    return check_buffers(ins, 5, outs, 2, inplace, 1);
}

int validate_resid_t(const dan_bf16 *r, const dan_bf16 *h, const dan_bf16 *gate, int64_t vs,
                     const dan_bf16 *r_out, int64_t B, int64_t T, int64_t D, bool *empty)
{
    if (B < 0 || T < 0 || D < 0) return DAN_EINVAL;
    if (D % 8 || D < 8) return DAN_EUNSUPPORTED;
    if (B > 0 && T > kMaxElems / B) return DAN_EINVAL;
    if (B * T > kMaxElems / D) return DAN_EINVAL;
    *empty = (B * T == 0);
    if (*empty) return DAN_OK;
    if (vs < D || vs > kMaxElems || (B - 1) > kMaxElems / vs) return DAN_EINVAL;
    if (vs % 8) return DAN_EALIGN;
    const int64_t bytes = B * T * D * 2;
    Buf ins[3] = {{r, span(r, bytes)}, {h, span(h, bytes)}, {gate, span(gate, vec_bytes(B, D, vs))}};
    Buf outs[1] = {{r_out, span(r_out, bytes)}};
    const int inplace[1][2] = {{0, 0}}; // r_out == r
    return check_buffers(ins, 3, outs, 1, inplace, 1);
}

int validate_ln_fp8(const dan_bf16 *x, const dan_bf16 *scale, const dan_bf16 *shift, int64_t vs,
                    float qscale, const uint8_t *q, int64_t B, int64_t T, int64_t D, float eps,
                    bool *empty)
{
    int st = check_rows(B, T, D, eps, vs, ln_d_ok(D));
    if (st == DAN_OK && !(std::isfinite(qscale) && qscale > 0.0f)) st = DAN_EINVAL;
    *empty = (st == DAN_OK && B * T == 0);
    if (st != DAN_OK || *empty) return st;
    Buf ins[3] = {{x, span(x, B * T * D * 2)}, {scale, span(scale, vec_bytes(B, D, vs))},
                  {shift, span(shift, vec_bytes(B, D, vs))}};
    Buf outs[1] = {{q, span(q, B * T * D)}}; // one byte per element; no in-place form
    return check_buffers(ins, 3, outs, 1, nullptr, 0);
}

int validate_qk(const dan_bf16 *const qkv[2][3], const int64_t Ts[2], const int64_t strides[2],
                int64_t heads, int64_t head_dim, const dan_bf16 *const w[4],
                const float *const rope[2], const float eps[2], const dan_bf16 *const outs_p[3],
                bool *empty)
{
    if (Ts[0] < 0 || Ts[1] < 0 || heads < 0 || head_dim < 0) return DAN_EINVAL;
    if (head_dim != 128 && head_dim != 64) return DAN_EUNSUPPORTED;
    if (heads < 1 || heads > (int64_t(1) << 20)) return DAN_EINVAL;
    if (!eps_ok(eps[0]) || !eps_ok(eps[1])) return DAN_EINVAL;
    const int64_t width = heads * head_dim;
    for (int s = 0; s < 2; ++s) {
        if (Ts[s] > kMaxElems / width) return DAN_EINVAL;
        if (Ts[s] > 0) {
            if (strides[s] < width || strides[s] > kMaxElems || Ts[s] > kMaxElems / strides[s])
                return DAN_EINVAL;
            if (strides[s] % 8) return DAN_EALIGN;
        }
    }
    const int64_t T = Ts[0] + Ts[1];
    *empty = (T == 0);
    if (*empty) return DAN_OK;

    Buf ins[14];
    int nin = 0;
    for (int s = 0; s < 2; ++s) {
        if (Ts[s] == 0) continue;
        const int64_t bytes = ((Ts[s] - 1) * strides[s] + width) * 2;
        for (int k = 0; k < 3; ++k) ins[nin++] = {qkv[s][k], span(qkv[s][k], bytes)};
        ins[nin++] = {w[2 * s], span(w[2 * s], head_dim * 2)};
        ins[nin++] = {w[2 * s + 1], span(w[2 * s + 1], head_dim * 2)};
        ins[nin++] = {rope[s], span(rope[s], Ts[s] * head_dim * 4)};
    }
    Buf outs[3];
    for (int k = 0; k < 3; ++k) outs[k] = {outs_p[k], span(outs_p[k], T * width * 2)};
    return check_buffers(ins, nin, outs, 3, nullptr, 0);
}

int launched(cudaError_t e) { return e == cudaSuccess ? DAN_OK : DAN_ECUDA; }

// The QK epilogue's arguments as the C entry points take them.
struct QkArgs {
    const dan_bf16 *q_txt, *k_txt, *v_txt;
    int64_t T_txt, txt_row_stride;
    const dan_bf16 *q_img, *k_img, *v_img;
    int64_t T_img, img_row_stride, heads, head_dim;
    const dan_bf16 *wq_txt, *wk_txt, *wq_img, *wk_img;
    const float *rope_txt, *rope_img;
    float eps_txt, eps_img;
    const dan_bf16 *q_out, *k_out, *v_out;
};

// Validate, and unless `check_only` launch, one QK epilogue call.
int qk_call(const QkArgs &a, bool neox, bool check_only, void *stream)
{
    const dan_bf16 *const qkv[2][3] = {{a.q_txt, a.k_txt, a.v_txt}, {a.q_img, a.k_img, a.v_img}};
    const int64_t Ts[2] = {a.T_txt, a.T_img}, strides[2] = {a.txt_row_stride, a.img_row_stride};
    const dan_bf16 *const w[4] = {a.wq_txt, a.wk_txt, a.wq_img, a.wk_img};
    const float *const rope[2] = {a.rope_txt, a.rope_img};
    const float eps[2] = {a.eps_txt, a.eps_img};
    const dan_bf16 *const outs[3] = {a.q_out, a.k_out, a.v_out};
    bool empty;
    const int st = validate_qk(qkv, Ts, strides, a.heads, a.head_dim, w, rope, eps, outs, &empty);
    if (st != DAN_OK || empty || check_only) return st;
    dan::QkProblem p;
    for (int s = 0; s < 2; ++s) {
        p.q[s] = qkv[s][0];
        p.k[s] = qkv[s][1];
        p.v[s] = qkv[s][2];
        p.T[s] = Ts[s];
        p.stride[s] = strides[s];
        p.wq[s] = w[2 * s];
        p.wk[s] = w[2 * s + 1];
        p.rope[s] = rope[s];
        p.eps[s] = eps[s];
    }
    p.q_out = const_cast<dan_bf16 *>(a.q_out);
    p.k_out = const_cast<dan_bf16 *>(a.k_out);
    p.v_out = const_cast<dan_bf16 *>(a.v_out);
    p.heads = a.heads;
    p.head_dim = a.head_dim;
    return launched(dan::launch_qk_norm_rope(p, neox, static_cast<cudaStream_t>(stream)));
}

} // namespace

namespace dan {

// The status word of each device the library runs on (a static device
// variable: one instance per device, never allocated by the library).
__device__ unsigned int g_device_status;

unsigned *device_status()
{
    static DeviceCache<unsigned *> cache;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return nullptr;
    return cached_per_device(cache, dev, []() -> unsigned * {
        void *ptr = nullptr;
        if (cudaGetSymbolAddress(&ptr, g_device_status) != cudaSuccess) return nullptr;
        return static_cast<unsigned *>(ptr);
    });
}

int sm_count()
{
    static DeviceCache<int> cache;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) dev = 0;
    return cached_per_device(cache, dev, [dev]() {
        int n = 0;
        if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n < 1)
            n = 1;
        return n;
    });
}

int max_smem_optin()
{
    static DeviceCache<int> cache;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) dev = 0;
    return cached_per_device(cache, dev, [dev]() {
        int v = 0;
        if (cudaDeviceGetAttribute(&v, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev) != cudaSuccess ||
            v <= 0)
            v = 48 * 1024;
        return v;
    });
}

cudaError_t allow_dynamic_smem(const void *fn, int smem)
{
    static std::mutex mu;
    static std::map<std::pair<const void *, int>, int> done; // (kernel, device) -> bytes set
    int dev = 0;
    const cudaError_t ge = cudaGetDevice(&dev);
    if (ge != cudaSuccess) return ge;
    std::lock_guard<std::mutex> lk(mu);
    auto it = done.find({fn, dev});
    if (it == done.end()) {
        // Every kernel asks for the largest shared-memory split of the SM's
        // on-chip memory, so consecutive launches of different kernels never
        // wait for the SM to change its L1 / shared split.
        const cudaError_t e = cudaFuncSetAttribute(
            fn, cudaFuncAttributePreferredSharedMemoryCarveout, (int)cudaSharedmemCarveoutMaxShared);
        if (e != cudaSuccess) return e;
        it = done.emplace(std::make_pair(fn, dev), 0).first;
    }
    if (smem > 48 * 1024 && it->second < smem) {
        const cudaError_t e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
        if (e != cudaSuccess) return e;
        it->second = smem;
    }
    return cudaSuccess;
}

} // namespace dan

extern "C" {

int dan_get_device_status(unsigned int *status)
{
    if (!status) return DAN_EINVAL;
    unsigned v = 0, zero = 0;
    if (cudaMemcpyFromSymbol(&v, dan::g_device_status, sizeof v) != cudaSuccess) return DAN_ECUDA;
    if (cudaMemcpyToSymbol(dan::g_device_status, &zero, sizeof zero) != cudaSuccess) return DAN_ECUDA;
    *status = v;
    return DAN_OK;
}

int dan_selftest_wait_timeout(unsigned long long limit_ns, void *stream)
{
    if (limit_ns == 0 || limit_ns > 2000000000ull) return DAN_EINVAL;
    if (!dan::device_status()) return DAN_ECUDA;
    return launched(dan::launch_wait_selftest(limit_ns, static_cast<cudaStream_t>(stream)));
}

const char *dan_status_string(int status)
{
    switch (status) {
    case DAN_OK: return "DAN_OK";
    case DAN_EINVAL: return "DAN_EINVAL: null pointer, negative size, bad stride or bad eps";
    case DAN_EUNSUPPORTED: return "DAN_EUNSUPPORTED: D or head_dim outside the supported set";
    case DAN_EALIGN: return "DAN_EALIGN: pointer or stride not 16-byte aligned";
    case DAN_EALIAS: return "DAN_EALIAS: an output overlaps an input or another output";
    case DAN_ECUDA: return "DAN_ECUDA: the kernel launch failed";
    default: return "unknown dan status";
    }
}

int dan_can_use_rms_modulate(const dan_bf16 *x, const dan_bf16 *weight, const dan_bf16 *scale,
                             const dan_bf16 *shift, int64_t vec_bstride, const dan_bf16 *y,
                             int64_t B, int64_t T, int64_t D, float eps)
{
    bool empty;
    return validate_rms(x, weight, scale, shift, vec_bstride, y, B, T, D, eps, &empty);
}

int dan_rms_modulate(const dan_bf16 *x, const dan_bf16 *weight, const dan_bf16 *scale,
                     const dan_bf16 *shift, int64_t vec_bstride, dan_bf16 *y, int64_t B, int64_t T,
                     int64_t D, float eps, void *stream)
{
    bool empty;
    const int st = validate_rms(x, weight, scale, shift, vec_bstride, y, B, T, D, eps, &empty);
    if (st != DAN_OK || empty) return st;
    dan::RowProblem p{x, nullptr, nullptr, weight, scale, shift, vec_bstride, y, nullptr,
                      B, T, D, eps};
    return launched(dan::launch_rms_modulate(p, static_cast<cudaStream_t>(stream)));
}

int dan_can_use_gated_rms_modulate(const dan_bf16 *r, const dan_bf16 *h, const dan_bf16 *gate,
                                   const dan_bf16 *weight, const dan_bf16 *scale,
                                   const dan_bf16 *shift, int64_t vec_bstride,
                                   const dan_bf16 *r_out, const dan_bf16 *y, int64_t B, int64_t T,
                                   int64_t D, float eps)
{
    bool empty;
    return validate_gated(r, h, gate, weight, scale, shift, vec_bstride, r_out, y, B, T, D, eps,
                          &empty);
}

int dan_gated_rms_modulate(const dan_bf16 *r, const dan_bf16 *h, const dan_bf16 *gate,
                           const dan_bf16 *weight, const dan_bf16 *scale, const dan_bf16 *shift,
                           int64_t vec_bstride, dan_bf16 *r_out, dan_bf16 *y, int64_t B, int64_t T,
                           int64_t D, float eps, void *stream)
{
    bool empty;
    const int st = validate_gated(r, h, gate, weight, scale, shift, vec_bstride, r_out, y, B, T, D,
                                  eps, &empty);
    if (st != DAN_OK || empty) return st;
    dan::RowProblem p{r, h, gate, weight, scale, shift, vec_bstride, y, r_out, B, T, D, eps};
    return launched(dan::launch_gated_rms_modulate(p, static_cast<cudaStream_t>(stream)));
}

int dan_can_use_ln_modulate(const dan_bf16 *x, const dan_bf16 *scale, const dan_bf16 *shift,
                            int64_t vec_bstride, const dan_bf16 *y, int64_t B, int64_t T,
                            int64_t D, float eps)
{
    bool empty;
    return validate_ln(x, scale, shift, vec_bstride, y, B, T, D, eps, &empty);
}

int dan_ln_modulate(const dan_bf16 *x, const dan_bf16 *scale, const dan_bf16 *shift,
                    int64_t vec_bstride, dan_bf16 *y, int64_t B, int64_t T, int64_t D, float eps,
                    void *stream)
{
    bool empty;
    const int st = validate_ln(x, scale, shift, vec_bstride, y, B, T, D, eps, &empty);
    if (st != DAN_OK || empty) return st;
    dan::RowProblem p{x, nullptr, nullptr, nullptr, scale, shift, vec_bstride, y, nullptr,
                      B, T, D, eps};
    return launched(dan::launch_ln_modulate(p, static_cast<cudaStream_t>(stream)));
}

int dan_can_use_gated_ln_modulate(const dan_bf16 *r, const dan_bf16 *h, const dan_bf16 *gate,
                                  const dan_bf16 *scale, const dan_bf16 *shift,
                                  int64_t vec_bstride, const dan_bf16 *r_out, const dan_bf16 *y,
                                  int64_t B, int64_t T, int64_t D, float eps)
{
    bool empty;
    return validate_gated_ln(r, h, gate, scale, shift, vec_bstride, r_out, y, B, T, D, eps,
                             &empty);
}

int dan_gated_ln_modulate(const dan_bf16 *r, const dan_bf16 *h, const dan_bf16 *gate,
                          const dan_bf16 *scale, const dan_bf16 *shift, int64_t vec_bstride,
                          dan_bf16 *r_out, dan_bf16 *y, int64_t B, int64_t T, int64_t D,
                          float eps, void *stream)
{
    bool empty;
    const int st = validate_gated_ln(r, h, gate, scale, shift, vec_bstride, r_out, y, B, T, D,
                                     eps, &empty);
    if (st != DAN_OK || empty) return st;
    dan::RowProblem p{r, h, gate, nullptr, scale, shift, vec_bstride, y, r_out, B, T, D, eps};
    return launched(dan::launch_gated_ln_modulate(p, static_cast<cudaStream_t>(stream)));
}

int dan_can_use_gated_residual_transposed(const dan_bf16 *r, const dan_bf16 *h,
                                          const dan_bf16 *gate, int64_t vec_bstride,
                                          const dan_bf16 *r_out, int64_t B, int64_t T, int64_t D)
{
    bool empty;
    return validate_resid_t(r, h, gate, vec_bstride, r_out, B, T, D, &empty);
}

int dan_gated_residual_transposed(const dan_bf16 *r, const dan_bf16 *h, const dan_bf16 *gate,
                                  int64_t vec_bstride, dan_bf16 *r_out, int64_t B, int64_t T,
                                  int64_t D, void *stream)
{
    bool empty;
    const int st = validate_resid_t(r, h, gate, vec_bstride, r_out, B, T, D, &empty);
    if (st != DAN_OK || empty) return st;
    const dan::ResidProblem p{r, h, gate, r_out, B, T, D, vec_bstride};
    return launched(dan::launch_gated_residual_transposed(p, static_cast<cudaStream_t>(stream)));
}

int dan_can_use_ln_modulate_fp8(const dan_bf16 *x, const dan_bf16 *scale, const dan_bf16 *shift,
                                int64_t vec_bstride, float qscale, const uint8_t *q, int64_t B,
                                int64_t T, int64_t D, float eps)
{
    bool empty;
    return validate_ln_fp8(x, scale, shift, vec_bstride, qscale, q, B, T, D, eps, &empty);
}

int dan_ln_modulate_fp8(const dan_bf16 *x, const dan_bf16 *scale, const dan_bf16 *shift,
                        int64_t vec_bstride, float qscale, uint8_t *q, int64_t B, int64_t T,
                        int64_t D, float eps, void *stream)
{
    bool empty;
    const int st = validate_ln_fp8(x, scale, shift, vec_bstride, qscale, q, B, T, D, eps, &empty);
    if (st != DAN_OK || empty) return st;
    dan::RowProblem p{x, nullptr, nullptr, nullptr, scale, shift, vec_bstride, nullptr, nullptr,
                      B, T, D, eps};
    p.q = q;
    p.qinv = 1.0f / qscale; // one IEEE division on the host: rn(1 / qscale)
    return launched(dan::launch_ln_modulate_fp8(p, static_cast<cudaStream_t>(stream)));
}

int dan_can_use_qk_norm_rope_epilogue(
    const dan_bf16 *q_txt, const dan_bf16 *k_txt, const dan_bf16 *v_txt, int64_t T_txt,
    int64_t txt_row_stride, const dan_bf16 *q_img, const dan_bf16 *k_img, const dan_bf16 *v_img,
    int64_t T_img, int64_t img_row_stride, int64_t heads, int64_t head_dim,
    const dan_bf16 *wq_txt, const dan_bf16 *wk_txt, const dan_bf16 *wq_img,
    const dan_bf16 *wk_img, const float *rope_txt, const float *rope_img, float eps_txt,
    float eps_img, const dan_bf16 *q_out, const dan_bf16 *k_out, const dan_bf16 *v_out)
{
    const QkArgs a{q_txt,  k_txt,  v_txt,    T_txt,    txt_row_stride, q_img,   k_img,   v_img,
                   T_img,  img_row_stride,   heads,    head_dim,       wq_txt,  wk_txt,  wq_img,
                   wk_img, rope_txt,         rope_img, eps_txt,        eps_img, q_out,   k_out,
                   v_out};
    return qk_call(a, false, true, nullptr);
}

int dan_qk_norm_rope_epilogue(const dan_bf16 *q_txt, const dan_bf16 *k_txt, const dan_bf16 *v_txt,
                              int64_t T_txt, int64_t txt_row_stride, const dan_bf16 *q_img,
                              const dan_bf16 *k_img, const dan_bf16 *v_img, int64_t T_img,
                              int64_t img_row_stride, int64_t heads, int64_t head_dim,
                              const dan_bf16 *wq_txt, const dan_bf16 *wk_txt,
                              const dan_bf16 *wq_img, const dan_bf16 *wk_img,
                              const float *rope_txt, const float *rope_img, float eps_txt,
                              float eps_img, dan_bf16 *q_out, dan_bf16 *k_out, dan_bf16 *v_out,
                              void *stream)
{
    const QkArgs a{q_txt,  k_txt,  v_txt,    T_txt,    txt_row_stride, q_img,   k_img,   v_img,
                   T_img,  img_row_stride,   heads,    head_dim,       wq_txt,  wk_txt,  wq_img,
                   wk_img, rope_txt,         rope_img, eps_txt,        eps_img, q_out,   k_out,
                   v_out};
    return qk_call(a, false, false, stream);
}

int dan_can_use_qk_norm_rope_neox_epilogue(
    const dan_bf16 *q_txt, const dan_bf16 *k_txt, const dan_bf16 *v_txt, int64_t T_txt,
    int64_t txt_row_stride, const dan_bf16 *q_img, const dan_bf16 *k_img, const dan_bf16 *v_img,
    int64_t T_img, int64_t img_row_stride, int64_t heads, int64_t head_dim,
    const dan_bf16 *wq_txt, const dan_bf16 *wk_txt, const dan_bf16 *wq_img,
    const dan_bf16 *wk_img, const float *rope_txt, const float *rope_img, float eps_txt,
    float eps_img, const dan_bf16 *q_out, const dan_bf16 *k_out, const dan_bf16 *v_out)
{
    const QkArgs a{q_txt,  k_txt,  v_txt,    T_txt,    txt_row_stride, q_img,   k_img,   v_img,
                   T_img,  img_row_stride,   heads,    head_dim,       wq_txt,  wk_txt,  wq_img,
                   wk_img, rope_txt,         rope_img, eps_txt,        eps_img, q_out,   k_out,
                   v_out};
    return qk_call(a, true, true, nullptr);
}

int dan_qk_norm_rope_neox_epilogue(const dan_bf16 *q_txt, const dan_bf16 *k_txt,
                                   const dan_bf16 *v_txt, int64_t T_txt, int64_t txt_row_stride,
                                   const dan_bf16 *q_img, const dan_bf16 *k_img,
                                   const dan_bf16 *v_img, int64_t T_img, int64_t img_row_stride,
                                   int64_t heads, int64_t head_dim, const dan_bf16 *wq_txt,
                                   const dan_bf16 *wk_txt, const dan_bf16 *wq_img,
                                   const dan_bf16 *wk_img, const float *rope_txt,
                                   const float *rope_img, float eps_txt, float eps_img,
                                   dan_bf16 *q_out, dan_bf16 *k_out, dan_bf16 *v_out, void *stream)
{
    const QkArgs a{q_txt,  k_txt,  v_txt,    T_txt,    txt_row_stride, q_img,   k_img,   v_img,
                   T_img,  img_row_stride,   heads,    head_dim,       wq_txt,  wk_txt,  wq_img,
                   wk_img, rope_txt,         rope_img, eps_txt,        eps_img, q_out,   k_out,
                   v_out};
    return qk_call(a, true, false, stream);
}

} // extern "C"
