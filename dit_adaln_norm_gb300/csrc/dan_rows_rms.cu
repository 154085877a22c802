// dan_rows_rms.cu -- launches of the RMSNorm + modulate row kernel.
#include "dan_rows.cuh"

namespace dan {

// Pipeline shapes (warps NW, warps per row TW, slots per team SPC), chosen
// by measurement: single-warp teams with two slots each, twelve of them
// when there are many rows per SM and eight otherwise, did better than
// fewer teams with more slots or multi-warp teams at these widths; rows of
// 6144 and 8192 are shared by three and four warps, which keeps them in
// registers.
cudaError_t launch_rms_modulate(const RowProblem &q, cudaStream_t s)
{
    switch (q.D) {
    case 2048: return launch_ring<kRms, 1, 8, 8, 1, 2, false>(q, s);
    case 4096: return many_rows(q) ? launch_ring<kRms, 2, 8, 12, 1, 2, false>(q, s)
                                   : launch_ring<kRms, 2, 8, 8, 1, 2, false>(q, s);
    case 6144: return launch_ring<kRms, 3, 8, 12, 3, 2, false>(q, s);
    default: return launch_ring<kRms, 4, 8, 16, 4, 1, false>(q, s); // 8192: 4 warps per row
    }
}

} // namespace dan
