// dan_ring.cuh -- warp-fed bulk-copy pipelines: mbarrier and cp.async.bulk
// primitives, the bounded wait, and the slot schedule shared by the kernels.
//
// Every warp of a CTA requests its own work units (whole rows, or a head
// group of one token) with 1-D bulk copies (cp.async.bulk, global ->
// shared, completion counted in bytes on an mbarrier) into SPC shared-memory
// slots that it alone uses.  Its i-th unit goes to slot i % SPC and
// completes phase (i / SPC) & 1 of that slot's barrier.  As soon as the
// warp has copied unit i out of its slot into registers it requests unit
// i + SPC into the same slot, so the copy overlaps its work on unit i.
// Nothing else waits on a warp's barriers and the warp waits on them in
// order, so a barrier is never more than one phase ahead of its waiter and
// the parity test cannot alias; no copy is left in flight when the warp
// finishes, because every unit it requests is one it then waits for.
//
// Every wait is bounded in time.  After the limit the waiter sets a bit in a
// device status word and returns; the host reads it with
// dan_get_device_status().
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

namespace dan {

// Status bits a kernel may set in the device status word.
constexpr unsigned kStatusWaitFull = 1u;  // a warp gave up waiting for a unit it requested
constexpr unsigned kStatusWaitDrain = 4u; // after that, it gave up waiting for its other copies

__device__ __forceinline__ unsigned smem_addr(const void *p)
{
    return (unsigned)__cvta_generic_to_shared(p);
}

__device__ __forceinline__ unsigned long long global_ns()
{
    unsigned long long t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

__device__ __forceinline__ void mbar_init(uint64_t *bar, unsigned count)
{
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_addr(bar)), "r"(count)
                 : "memory");
}

// Make barrier initialisation visible to the bulk-copy (async) proxy.
__device__ __forceinline__ void mbar_init_fence()
{
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

// Arrive once and expect `bytes` of bulk-copy completion in this phase.
__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t *bar, unsigned bytes)
{
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_addr(bar)),
                 "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t *bar, unsigned parity)
{
    unsigned ok;
    asm volatile("{\n\t.reg .pred p;\n\t"
                 "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
                 "selp.u32 %0, 1, 0, p;\n\t}"
                 : "=r"(ok)
                 : "r"(smem_addr(bar)), "r"(parity)
                 : "memory");
    return ok != 0;
}

// Wait for the completion of the phase of `bar` with parity `parity`;
// false if it has not completed within `limit_ns` nanoseconds.  An
// iteration cap backs up the clock (each try_wait may itself suspend for a
// while, so the clock ends every wait long before the cap in practice).
__device__ __forceinline__ bool mbar_wait(uint64_t *bar, unsigned parity,
                                          unsigned long long limit_ns)
{
    if (mbar_try_wait(bar, parity)) return true;
    const unsigned long long t0 = global_ns();
#pragma unroll 1
    for (unsigned it = 0; it < (1u << 20); ++it) {
#pragma unroll 1
        for (int i = 0; i < 32; ++i)
            if (mbar_try_wait(bar, parity)) return true;
        if (global_ns() - t0 > limit_ns) return false;
    }
    return false;
}

__device__ __forceinline__ void mbar_arrive(uint64_t *bar)
{
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_addr(bar)) : "memory");
}

// 1-D bulk copy global -> shared of `bytes` (multiple of 16, both addresses
// 16-byte aligned) completing on `bar`.
__device__ __forceinline__ void bulk_load(void *smem_dst, const void *gmem_src, unsigned bytes,
                                          uint64_t *bar)
{
    asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes "
                 "[%0], [%1], %2, [%3];" ::"r"(smem_addr(smem_dst)),
                 "l"(gmem_src), "r"(bytes), "r"(smem_addr(bar))
                 : "memory");
}

// Hint the L2 to fetch `bytes` (a multiple of 16, 16-byte aligned) of
// global memory.  It returns nothing to the SM, so it may run before the
// dependency wait on data the previous grid is still writing: the L2 is the
// point of coherence, a write reaching a line after (or while) it is filled
// leaves the written data in it, and every read of the data still happens
// after the wait.
__device__ __forceinline__ void prefetch_l2(const void *gmem, unsigned bytes)
{
    asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(gmem), "r"(bytes) : "memory");
}

// The same hint for the cache line holding one address (no alignment).
__device__ __forceinline__ void prefetch_l2_line(const void *gmem)
{
    asm volatile("prefetch.global.L2 [%0];" ::"l"(gmem) : "memory");
}

// After a warp's generic-proxy reads of a slot, order them before the next
// bulk copy (async proxy) into it: every reading lane fences, then the warp
// converges, and lane 0 may issue the refill (measured: without the fence a
// refill occasionally overwrote a slot still being read).  All 32 lanes
// must call this.
__device__ __forceinline__ void slot_reads_done()
{
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
    __syncwarp();
}

// Programmatic dependent launch.  A kernel launched with programmatic stream
// serialization (launch_overlapped) may start while the grid before it in
// the stream is still running; every thread calls grid_dependency_wait()
// before its first global-memory access, which returns once that grid has
// completed and its writes are visible (at once when there is none).
// allow_dependents() lets the next such grid start the same way.
__device__ __forceinline__ void grid_dependency_wait()
{
    asm volatile("griddepcontrol.wait;" ::: "memory");
}

__device__ __forceinline__ void allow_dependents()
{
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

__device__ __forceinline__ void set_status(unsigned *status, unsigned bit)
{
    if (status) atomicOr(status, bit);
}

// Slot and barrier phase of a warp's i-th unit (see the header comment).
template <int SPC>
struct WarpPipe {
    __device__ __forceinline__ static int slot(int i) { return i % SPC; }
    __device__ __forceinline__ static unsigned phase(int i) { return (unsigned)(i / SPC) & 1u; }

    // Wait for unit i on the warp's barriers `full` (SPC of them).
    __device__ __forceinline__ static bool wait(uint64_t *full, int i, unsigned long long limit_ns)
    {
        return mbar_wait(full + slot(i), phase(i), limit_ns);
    }

    // Failure path, after the wait for unit i ran out: wait (bounded again)
    // for every unit the warp has requested and not consumed, i .. i+SPC-1
    // below `units`, so that no copy lands after the CTA has exited; record
    // the failure.  Returns the status bits set.
    __device__ static unsigned abort(uint64_t *full, int i, int units, unsigned *status,
                                     unsigned long long limit_ns)
    {
        unsigned bits = kStatusWaitFull;
        for (int u = i; u < i + SPC && u < units; ++u)
            if (!wait(full, u, limit_ns)) {
                bits |= kStatusWaitDrain;
                break;
            }
        set_status(status, bits);
        return bits;
    }
};

} // namespace dan
