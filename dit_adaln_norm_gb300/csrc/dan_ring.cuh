// dan_ring.cuh -- TMA bulk-copy row ring: mbarrier and cp.async.bulk
// primitives, the bounded wait, and the slot schedule shared by the kernels.
//
// One producer thread per CTA issues 1-D bulk copies (cp.async.bulk, global
// -> shared, completion counted in bytes on an mbarrier) of whole rows into
// a ring of shared-memory slots, in row order, so rows land roughly in the
// order they are consumed; consumer warps take rows from the ring.
//
// Slot ownership: consumer warp c owns slots c, c + NC, ..., c + NC*(SPC-1)
// and takes the CTA's rows c, c + NC, c + 2NC, ...; its i-th row lives in
// slot c + NC*(i % SPC) in phase (i / SPC) & 1.  A slot is therefore only
// ever used by one consumer, which consumed its previous phase itself: a
// barrier is never two phases behind its waiter, so the parity test cannot
// alias.  The producer refills a slot only after its consumer released it,
// so each slot has at most one copy in flight; before the CTA exits the
// producer waits for the last copy it issued into every slot.
//
// Every wait is bounded in time.  After the limit the waiter sets a bit in a
// device status word and returns; the host reads it with
// dan_get_device_status().
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

namespace dan {

// Status bits a kernel may set in the device status word.
constexpr unsigned kStatusWaitFull = 1u;  // a consumer gave up waiting for a row
constexpr unsigned kStatusWaitEmpty = 2u; // the producer gave up waiting for a slot
constexpr unsigned kStatusWaitDrain = 4u; // the producer gave up waiting for its own copies

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

__device__ __forceinline__ void mbar_arrive(uint64_t *bar)
{
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_addr(bar)) : "memory");
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

// A consumer's release of a slot: its generic-proxy reads of the slot must
// be ordered before the producer's next bulk copy (async proxy) into it,
// which needs a proxy fence by every reading thread before the arrive
// (measured: without it a refill occasionally overwrote a slot still being
// read).  All 32 lanes must call this.
__device__ __forceinline__ void ring_release(uint64_t *empty_slot, int lane)
{
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
    __syncwarp();
    if (lane == 0) mbar_arrive(empty_slot);
}

__device__ __forceinline__ void set_status(unsigned *status, unsigned bit)
{
    if (status) atomicOr(status, bit);
}

// Slot and phase of the i-th row of consumer c (see the header comment).
template <int NC, int SPC>
struct RingSchedule {
    static constexpr int S = NC * SPC;
    __device__ __forceinline__ static int slot(int c, int i) { return c + NC * (i % SPC); }
    __device__ __forceinline__ static unsigned phase(int i) { return (unsigned)(i / SPC) & 1u; }
};

// Producer side for `n` rows: row k belongs to consumer k % NC as its
// (k / NC)-th row.  `issue(k, slot)` must arm and issue the copies of row k
// into `slot` (one mbar_arrive_expect_tx on full[slot] with the total bytes,
// then the bulk copies).  Returns after the last copy of every slot landed,
// with the status bits it set (0 when every wait completed).
template <int NC, int SPC, typename Issue>
__device__ __forceinline__ unsigned ring_produce(int n, uint64_t *full, uint64_t *empty,
                                                 unsigned *status, unsigned long long limit_ns,
                                                 Issue issue)
{
    using R = RingSchedule<NC, SPC>;
    unsigned failed = 0;
    int issued = 0;
    for (int k = 0; k < n; ++k) {
        const int c = k % NC, i = k / NC, s = R::slot(c, i);
        if (i >= SPC && !mbar_wait(empty + s, R::phase(i - SPC), limit_ns)) {
            set_status(status, kStatusWaitEmpty);
            failed |= kStatusWaitEmpty;
            break;
        }
        issue(k, s);
        issued = k + 1;
    }
    // drain: the last copy issued into each slot (earlier ones have landed,
    // since a slot is refilled only after its consumer released it)
    for (int k = issued - 1; k >= 0 && k >= issued - R::S; --k) {
        const int c = k % NC, i = k / NC;
        if (!mbar_wait(full + R::slot(c, i), R::phase(i), limit_ns)) {
            set_status(status, kStatusWaitDrain);
            failed |= kStatusWaitDrain;
            break;
        }
    }
    return failed;
}

} // namespace dan
