// dan_noalloc.cu -- dan_rms_modulate_noalloc: the RMS + modulate kernel for
// callers that cannot allocate device memory, with its scratch (one
// bounded-wait failure record per CTA) in a static device array.
#include "../../include/dan.h"
#include "dan_rows.cuh"

namespace dan {
namespace {

// Maximum number of CTAs a call may launch: one record each (1 KB).  The
// launch uses one CTA per SM (at most the row count), so this bounds the
// GPU's SM count, not the problem size.
constexpr int kNoAllocMaxCtas = 256;

// Shared by every call on a device and kept until the process exits; each
// CTA clears its own record when it starts.  The records are internal: a
// caller sees a failed wait through the device status word
// (dan_get_device_status), which the same kernels also set.
static __device__ __align__(256) unsigned int g_noalloc_scratch[kNoAllocMaxCtas];

// Device address of the scratch array for the current device, looked up
// once per device (host code cannot use the symbol itself as an address).
unsigned *noalloc_scratch()
{
    static DeviceCache<unsigned *> cache;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return nullptr;
    return cached_per_device(cache, dev, []() -> unsigned * {
        void *ptr = nullptr;
        if (cudaGetSymbolAddress(&ptr, g_noalloc_scratch) != cudaSuccess) return nullptr;
        return static_cast<unsigned *>(ptr);
    });
}

} // namespace
} // namespace dan

extern "C" int dan_rms_modulate_noalloc(const dan_bf16 *x, const dan_bf16 *weight,
                                        const dan_bf16 *scale, const dan_bf16 *shift,
                                        int64_t vec_bstride, dan_bf16 *y, int64_t B, int64_t T,
                                        int64_t D, float eps, void *stream)
{
    const int st = dan_can_use_rms_modulate(x, weight, scale, shift, vec_bstride, y, B, T, D, eps);
    if (st != DAN_OK || B * T == 0) return st;
    if (dan::ring_grid(B * T) > dan::kNoAllocMaxCtas) return DAN_EUNSUPPORTED; // records run out
    unsigned *scratch = dan::noalloc_scratch();
    if (!scratch) return DAN_ECUDA;
    dan::RowProblem q{x, nullptr, nullptr, weight, scale, shift, vec_bstride, y, nullptr,
                      B, T, D, eps};
    // the shapes of dan_rms_modulate; the launcher checks its grid against
    // the record capacity again before launching
    const cudaError_t e = dan::launch_rms_shapes<true>(q, static_cast<cudaStream_t>(stream),
                                                       scratch, dan::kNoAllocMaxCtas);
    return e == cudaSuccess ? DAN_OK : DAN_ECUDA;
}
