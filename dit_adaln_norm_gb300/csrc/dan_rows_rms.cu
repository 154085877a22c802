// dan_rows_rms.cu -- launches of the RMSNorm + modulate ring kernel.
#include "dan_rows.cuh"

namespace dan {

// Pipeline shapes (warps NW, slots per warp SPC), chosen by measurement:
// eight warps did better than fewer with more slots each, or more warps
// (which also cap the registers a row needs).
cudaError_t launch_rms_modulate(const RowProblem &q, cudaStream_t s)
{
    switch (q.D) {
    case 2048: return launch_ring<kRms, 1, 8, 8, 2, false>(q, s);
    case 4096: return launch_ring<kRms, 2, 8, 8, 2, false>(q, s);
    case 6144: return launch_ring<kRms, 3, 8, 8, 1, false>(q, s);
    default: return launch_ring<kRms, 4, 8, 8, 1, false>(q, s); // 8192
    }
}

} // namespace dan
