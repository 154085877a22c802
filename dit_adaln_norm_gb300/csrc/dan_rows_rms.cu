// dan_rows_rms.cu -- launches of the RMSNorm + modulate row kernel (the
// shapes per width are launch_rms_shapes in dan_rows.cuh).
#include "dan_rows.cuh"

namespace dan {

cudaError_t launch_rms_modulate(const RowProblem &q, cudaStream_t s)
{
    return launch_rms_shapes<false>(q, s);
}

} // namespace dan
