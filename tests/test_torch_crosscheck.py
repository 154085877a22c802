"""Informational cross-check against torch eager (not a parity gate).

The library defines its own reduction order and a defined rsqrt, so its bits
are not torch's.  This measures how far they are apart at the metric shape:
the fraction of output elements with identical bits and the largest
difference, in bf16 units in the last place of the larger addend of the
final sum (max(|p|, |shift|), p = bf16(n * bf16(1 + scale))), for LayerNorm
and RMSNorm followed by the eager modulate chain y = bf16(p + shift).  The
bounds asserted are loose; the measured values are printed (run with -s)
and recorded with the design notes."""
import numpy as np
import pytest
import torch
import torch.nn.functional as F

from dit_adaln_norm_gb300 import ops, synth
from _gpu import to_dev

pytestmark = pytest.mark.gpu
EPS = 1e-6
T, D = 4216, 4096


def _ordered(bits: np.ndarray) -> np.ndarray:
    """bf16 bit patterns as integers whose order is the values' order."""
    b = bits.astype(np.int32) & 0xFFFF
    return np.where(b & 0x8000, 0x8000 - b, b)


def _compare(ours: torch.Tensor, ref: torch.Tensor, p: torch.Tensor, shift: torch.Tensor):
    a = ours.cpu().view(torch.int16).numpy()
    b = ref.cpu().view(torch.int16).numpy()
    same = float(np.mean(_ordered(a) == _ordered(b)))
    diff = (ours.float() - ref.float()).abs().cpu().numpy()
    big = torch.maximum(p.float().abs(), shift.float().abs().expand_as(p)).cpu().numpy()
    ulp = np.exp2(np.floor(np.log2(np.maximum(big, 2.0 ** -126))) - 7)  # bf16 ulp at big
    return same, float((diff / ulp).max())


@pytest.mark.parametrize("kind", ["ln", "rms"])
def test_against_torch_eager(kind):
    x = to_dev(synth.outlier_rows_bf16((1, T, D), synth.SEED_X, synth.SEED_OUTLIER))
    vec = to_dev(synth.normal_bf16((1, 6 * D), synth.SEED_VEC, 0.2))
    sc, sh = vec[:, :D], vec[:, D:2 * D]
    if kind == "ln":
        ours = ops.ln_modulate(x, sc, sh, EPS)
        n = F.layer_norm(x, (D,), eps=EPS)
    else:
        ours = ops.rms_modulate(x, sc, sh, EPS)
        n = F.rms_norm(x, (D,), eps=EPS)
    p = n * (1 + sc[:, None, :])  # bf16 aten ops, each rounded
    ref = p + sh[:, None, :]
    same, worst = _compare(ours, ref, p, sh[:, None, :])
    print(f"\n{kind}: {same * 100:.4f}% of elements bit-identical to torch eager, "
          f"max difference {worst:.2f} bf16 ulp of the larger addend")
    assert same > 0.99 and worst <= 4
