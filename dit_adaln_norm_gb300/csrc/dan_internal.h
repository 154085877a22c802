// dan_internal.h -- launch interface between the C-ABI shim and the kernels.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include <atomic>

namespace dan {

// Per-device caches of values that never change once known (an SM count,
// a device symbol's address).  Entries are atomics: host threads that race
// on a device's first use each compute the same value and store it.
// Devices beyond the table are served uncached.
constexpr int kCachedDevices = 64;

template <typename T>
using DeviceCache = std::atomic<T>[kCachedDevices];

// cache[dev], computing it with compute() the first time; a result equal to
// T{} (a failed lookup) is returned but not cached.
template <typename T, typename F>
T cached_per_device(DeviceCache<T> &cache, int dev, F compute)
{
    if (dev < 0 || dev >= kCachedDevices) return compute();
    T v = cache[dev].load(std::memory_order_relaxed);
    if (v == T{}) {
        v = compute();
        if (v != T{}) cache[dev].store(v, std::memory_order_relaxed);
    }
    return v;
}

// One row problem: [B, T, D] rows, per-batch vectors with batch stride vs
// (elements), optional weight [D].  Arguments are validated by the shim.
struct RowProblem {
    const void *x;      // input rows (r for the gated form)
    const void *h;      // gated update rows, or nullptr
    const void *gate;   // per-batch gate, or nullptr
    const void *weight; // [D] or nullptr
    const void *scale;
    const void *shift;
    int64_t vs;
    void *y;
    void *r_out; // gated residual output, or nullptr
    int64_t B, T, D;
    float eps;
    void *q = nullptr;  // E4M3 output (LayerNorm + FP8), or nullptr
    float qinv = 0.0f;  // rn(1 / qscale) (LayerNorm + FP8)
};

struct QkProblem {
    const void *q[2], *k[2], *v[2]; // [0] text, [1] image
    int64_t T[2];
    int64_t stride[2]; // row stride in elements
    const void *wq[2], *wk[2];
    const float *rope[2];
    float eps[2];
    void *q_out, *k_out, *v_out;
    int64_t heads;
    int64_t head_dim; // 128 or 64
};

// Launch fn<<<grid, block, smem, s>>>(args...) with programmatic stream
// serialization: the grid may be scheduled before the previous grid in the
// stream has finished, so its kernel must begin with grid_dependency_wait()
// (dan_ring.cuh).  This hides the launch and the prologue behind the tail of
// the previous kernel; the order of memory accesses is unchanged.
template <typename... KArgs, typename... Args>
cudaError_t launch_overlapped(void (*fn)(KArgs...), int grid, int block, int smem, cudaStream_t s,
                              Args... args)
{
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)grid);
    cfg.blockDim = dim3((unsigned)block);
    cfg.dynamicSmemBytes = (size_t)smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, fn, args...);
}

// Residual gating in the [B, hidden, tokens] layout: r, r_out [B, D, T],
// h [B, T, D], gate [B, D] with batch stride vs.  Validated by the shim.
struct ResidProblem {
    const void *r, *h, *gate;
    void *r_out;
    int64_t B, T, D, vs;
};

cudaError_t launch_gated_residual_transposed(const ResidProblem &p, cudaStream_t s);

cudaError_t launch_rms_modulate(const RowProblem &p, cudaStream_t s);
cudaError_t launch_gated_rms_modulate(const RowProblem &p, cudaStream_t s);
cudaError_t launch_ln_modulate(const RowProblem &p, cudaStream_t s);
cudaError_t launch_ln_modulate_fp8(const RowProblem &p, cudaStream_t s);
cudaError_t launch_gated_ln_modulate(const RowProblem &p, cudaStream_t s);
// neox: rotate the halves' pairs (i, i + head_dim/2) instead of (2i, 2i+1).
cudaError_t launch_qk_norm_rope(const QkProblem &p, bool neox, cudaStream_t s);

// Number of SMs of the current device (cached per device).
int sm_count();

// Largest dynamic shared memory a block may opt in to on the current device.
int max_smem_optin();

// Let kernel `fn` use `smem` bytes of dynamic shared memory on the current
// device, and prefer the largest shared-memory carveout (each attribute set
// once per kernel and device, thread-safe).
cudaError_t allow_dynamic_smem(const void *fn, int smem);

// Device address of the current device's status word, where kernels record
// bounded-wait failures (cached per device; nullptr if it cannot be had).
unsigned *device_status();

// Launch the bounded-wait self-test kernel (see dan_selftest_wait_timeout).
cudaError_t launch_wait_selftest(unsigned long long limit_ns, cudaStream_t s);

} // namespace dan
