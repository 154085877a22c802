"""Helpers for the GPU parity tests: move bf16 bit patterns between numpy and
CUDA tensors, guard-banded outputs, and NaN-aware bitwise comparison."""
import numpy as np
import torch

from dit_adaln_norm_gb300 import synth

GUARD = 4096  # elements of sentinel before and after every guarded output
SENTINEL = 0x5A5A


def to_dev(bits: np.ndarray) -> torch.Tensor:
    """uint16 bf16 bits (any strides) -> contiguous CUDA bfloat16 tensor."""
    a = np.ascontiguousarray(bits).view(np.int16)
    return torch.from_numpy(a).view(torch.bfloat16).cuda()


def from_dev(t: torch.Tensor) -> np.ndarray:
    return t.contiguous().view(torch.int16).cpu().numpy().view(np.uint16)


def guarded(shape, device="cuda"):
    """An output tensor of `shape` inside a buffer whose GUARD elements on each
    side hold SENTINEL; check_guard() later verifies nothing was written there."""
    n = int(np.prod(shape))
    buf = torch.full((n + 2 * GUARD,), SENTINEL, dtype=torch.int16, device=device)
    view = buf[GUARD:GUARD + n].view(torch.bfloat16).view(*shape)
    return buf, view


def check_guard(buf):
    b = buf.cpu().numpy()
    assert np.all(b[:GUARD] == SENTINEL) and np.all(b[-GUARD:] == SENTINEL), "guard band written"


def is_nan_bits(b):
    return (b & 0x7FFF) > 0x7F80


def assert_bits_equal(got: np.ndarray, want: np.ndarray, what=""):
    got = np.asarray(got, np.uint16)
    want = np.asarray(want, np.uint16)
    assert got.shape == want.shape, (got.shape, want.shape)
    same = (got == want) | (is_nan_bits(got) & is_nan_bits(want))
    if not same.all():
        idx = np.argwhere(~same)
        first = [tuple(int(v) for v in i) for i in idx[:5]]
        vals = [(hex(int(got[tuple(i)])), hex(int(want[tuple(i)]))) for i in idx[:5]]
        raise AssertionError(f"{what}: {int((~same).sum())} of {same.size} elements differ; "
                             f"first at {first}: (gpu, oracle) = {vals}")


def adaln(B, D, n, seed, std, chunks=6):
    """Host views and device views of n per-batch vectors taken as chunks of
    one [B, chunks*D] embedding (batch stride chunks*D)."""
    emb = synth.normal_bf16((B, chunks * D), seed, std)
    E = to_dev(emb)
    host = [emb[:, i * D:(i + 1) * D] for i in range(n)]
    dev = [E[:, i * D:(i + 1) * D] for i in range(n)]
    return host, dev
