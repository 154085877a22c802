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
// CTA clears its own record when it starts.
static __device__ __align__(256) unsigned int g_noalloc_scratch[kNoAllocMaxCtas];

// Device address of the scratch array for the current device, looked up
// once per device (host code cannot use the symbol itself as an address).
unsigned *noalloc_scratch()
{
    static unsigned *cache[64] = {nullptr};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return nullptr;
    unsigned *&c = cache[dev & 63];
    if (c == nullptr) {
        void *ptr = nullptr;
        if (cudaGetSymbolAddress(&ptr, g_noalloc_scratch) != cudaSuccess) return nullptr;
        c = static_cast<unsigned *>(ptr);
    }
    return c;
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
    const int64_t rows = B * T;
    const int grid = (int)(rows < dan::sm_count() ? rows : dan::sm_count());
    if (grid > dan::kNoAllocMaxCtas) return DAN_EUNSUPPORTED; // more CTAs than scratch records
    unsigned *scratch = dan::noalloc_scratch();
    if (!scratch) return DAN_ECUDA;
    dan::RowProblem q{x, nullptr, nullptr, weight, scale, shift, vec_bstride, y, nullptr,
                      B, T, D, eps};
    const cudaStream_t s = static_cast<cudaStream_t>(stream);
    cudaError_t e;
    switch (D) {
    // the shapes of dan_rms_modulate, with a failure record per CTA
    case 2048: e = dan::launch_ring<dan::kRms, 1, 8, 8, 1, 2, false, true>(q, s, scratch); break;
    case 4096:
        e = dan::many_rows(q) ? dan::launch_ring<dan::kRms, 2, 8, 12, 1, 2, false, true>(q, s, scratch)
                              : dan::launch_ring<dan::kRms, 2, 8, 8, 1, 2, false, true>(q, s, scratch);
        break;
    case 6144: e = dan::launch_ring<dan::kRms, 3, 8, 12, 3, 2, false, true>(q, s, scratch); break;
    default: e = dan::launch_ring<dan::kRms, 4, 8, 16, 4, 1, false, true>(q, s, scratch); break;
    }
    return e == cudaSuccess ? DAN_OK : DAN_ECUDA;
}
