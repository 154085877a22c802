// dan_rows_gated.cu -- launches of the gated-residual RMSNorm + modulate ring
// kernel.
#include "dan_rows.cuh"

namespace dan {

cudaError_t launch_gated_rms_modulate(const RowProblem &q, cudaStream_t s)
{
    switch (q.D) {
    case 2048: return launch_ring<kGated, 1, 8, 8, 1, false>(q, s);
    case 4096: return launch_ring<kGated, 2, 8, 8, 1, false>(q, s);
    case 6144: return launch_ring<kGated, 3, 8, 4, 1, false>(q, s);
    default: return launch_ring<kGated, 4, 8, 4, 1, false>(q, s); // 8192
    }
}

} // namespace dan
