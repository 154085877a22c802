// dan_rows_lnfp8.cu -- launches of the LayerNorm + modulate + static FP8
// (E4M3) quantisation row kernel: the LayerNorm kernel with the quantised
// store ("SGLang diffusion fused-op package guide", list of fused producers:
// FLUX.2's LayerNorm, adaLN modulate and static FP8 quantisation in one
// kernel).
#include "dan_rows.cuh"

namespace dan {

cudaError_t launch_ln_modulate_fp8(const RowProblem &q, cudaStream_t s)
{
    return (q.D % 1024) ? launch_ln_fpt<kLnFp8, true>(q, s) : launch_ln_fpt<kLnFp8, false>(q, s);
}

} // namespace dan
