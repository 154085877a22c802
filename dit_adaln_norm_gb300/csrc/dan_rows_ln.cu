// dan_rows_ln.cu -- launches of the LayerNorm + modulate row kernel, and
// the bounded-wait self-test kernel.
#include "dan_rows.cuh"

namespace dan {

// ------------------------------------------------- bounded-wait self-test

// One warp waits on an mbarrier that nothing completes, through the same
// bounded wait the row kernels use, and records the timeout.
__global__ void wait_selftest_kernel(unsigned *status, unsigned long long limit_ns)
{
    __shared__ uint64_t bar;
    if (threadIdx.x == 0) {
        mbar_init(&bar, 1);
        mbar_init_fence();
    }
    __syncwarp();
    if (threadIdx.x == 0 && !mbar_wait(&bar, 0, limit_ns)) set_status(status, kStatusWaitFull);
}

cudaError_t launch_wait_selftest(unsigned long long limit_ns, cudaStream_t s)
{
    wait_selftest_kernel<<<1, 32, 0, s>>>(device_status(), limit_ns);
    return cudaGetLastError();
}

cudaError_t launch_ln_modulate(const RowProblem &q, cudaStream_t s)
{
    return (q.D % 1024) ? launch_ln_fpt<kLn, true>(q, s) : launch_ln_fpt<kLn, false>(q, s);
}

} // namespace dan
