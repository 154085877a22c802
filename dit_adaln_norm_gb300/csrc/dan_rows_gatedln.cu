// dan_rows_gatedln.cu -- launches of the gated residual + LayerNorm +
// modulate row kernel: r' = bf16(r + bf16(gate * h)) is stored, then the
// LayerNorm + modulate of r' ("SGLang diffusion fused-op package guide",
// residual variant; the LayerNorm of "PR #34126 report").
#include "dan_rows.cuh"

namespace dan {
namespace {

// A slot holds r and h (twice a LayerNorm slot), so wide rows get fewer
// slots than the plain LayerNorm.  With many rows each CTA takes every G-th
// row (against a contiguous block per CTA: 14.95 against 15.02 and 14.98
// against 15.30 us at [1,4096,3072], 20.99 against 21.02 and 20.89 against
// 21.16 at [1,4216,4096], on two GB300s).
template <bool RAGGED>
cudaError_t launch_gated_ln_fpt(const RowProblem &q, cudaStream_t s)
{
    switch ((q.D + 1023) / 1024) {
    case 1: return launch_ring<kGatedLn, 4, 1, 8, 1, 1, RAGGED>(q, s);
    case 2: return launch_ring<kGatedLn, 4, 2, 8, 1, 1, RAGGED>(q, s);
    case 3: return many_rows(q) ? launch_ring<kGatedLn, 4, 3, 12, 1, 1, RAGGED, false, 0, 0, 1, true>(q, s)
                                : launch_ring<kGatedLn, 4, 3, 8, 1, 1, RAGGED>(q, s);
    case 4: return many_rows(q) ? launch_ring<kGatedLn, 4, 4, 12, 1, 1, RAGGED, false, 0, 0, 1, true>(q, s)
                                : launch_ring<kGatedLn, 4, 4, 8, 1, 1, RAGGED>(q, s);
    case 5: return launch_ring<kGatedLn, 4, 5, 8, 2, 1, RAGGED>(q, s);
    case 6: return launch_ring<kGatedLn, 4, 6, 8, 2, 1, RAGGED>(q, s);
    case 7: return launch_ring<kGatedLn, 4, 7, 8, 2, 1, RAGGED>(q, s);
    default: return launch_ring<kGatedLn, 4, 8, 8, 2, 1, RAGGED>(q, s);
    }
}

} // namespace

cudaError_t launch_gated_ln_modulate(const RowProblem &q, cudaStream_t s)
{
    return (q.D % 1024) ? launch_gated_ln_fpt<true>(q, s) : launch_gated_ln_fpt<false>(q, s);
}

} // namespace dan
