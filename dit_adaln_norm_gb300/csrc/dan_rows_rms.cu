// dan_rows_rms.cu -- launches of the RMSNorm + modulate ring kernel.
#include "dan_rows.cuh"

namespace dan {

// Ring shapes (consumers NC, slots per consumer SPC): eight 8-16 KB slots
// per SM for rows up to 4096, four 16-32 KB ones above.
cudaError_t launch_rms_modulate(const RowProblem &q, cudaStream_t s)
{
    switch (q.D) {
    case 2048: return launch_ring<kRms, 1, 8, 8, 1, false>(q, s);
    case 4096: return launch_ring<kRms, 2, 8, 8, 1, false>(q, s);
    case 6144: return launch_ring<kRms, 3, 8, 4, 2, false>(q, s);
    default: return launch_ring<kRms, 4, 8, 4, 2, false>(q, s); // 8192
    }
}

} // namespace dan
