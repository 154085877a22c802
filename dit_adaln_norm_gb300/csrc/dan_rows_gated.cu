// dan_rows_gated.cu -- launches of the gated-residual RMSNorm + modulate row
// kernel.
#include "dan_rows.cuh"

namespace dan {

// Pipeline shapes (warps NW, warps per row TW, slots per team SPC), chosen
// by measurement at D = 4096 and 8192 and by the shared memory left for
// larger rows; a slot holds r and h.  Each CTA takes every G-th row
// (measured faster than contiguous blocks: 20.80 against 20.92 us at
// [1,4216,4096], 43.48 against 43.98 at [1,4216,8192]).
cudaError_t launch_gated_rms_modulate(const RowProblem &q, cudaStream_t s)
{
    switch (q.D) {
    case 2048: return launch_ring<kGated, 1, 8, 8, 1, 2, false, false, 0, 0, 1, true>(q, s);
    case 4096: return many_rows(q) ? launch_ring<kGated, 2, 8, 12, 1, 1, false, false, 0, 0, 1, true>(q, s)
                                   : launch_ring<kGated, 2, 8, 8, 1, 1, false, false, 0, 0, 1, true>(q, s);
    case 6144: return launch_ring<kGated, 3, 8, 6, 3, 1, false, false, 0, 0, 1, true>(q, s);
    default: // 8192: 2 warps per row, three rows per team prefetched before the wait
        return launch_ring<kGated, 4, 8, 6, 2, 1, false, false, 3, 0, 1, true>(q, s);
    }
}

} // namespace dan
