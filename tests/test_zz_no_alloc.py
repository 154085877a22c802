"""dan_rms_modulate_noalloc through the C ABI: the variant for callers that
cannot allocate device memory keeps its scratch in static device memory and
must give exactly the output of dan_rms_modulate, call after call (the
shared scratch keeps the previous call's contents).  Collected last."""
import numpy as np
import pytest
import torch

from dit_adaln_norm_gb300 import build as dan_build
from dit_adaln_norm_gb300 import ops, synth

pytestmark = pytest.mark.gpu
EPS = 1e-6


def _dev(bits):
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16).cuda()


@pytest.mark.parametrize("D,weight", [(4096, False), (2048, True)])
def test_noalloc_matches_rms_modulate_twice(D, weight):
    dan_build.build()
    lib = ops.load()
    B, T = 2, 1500
    x = _dev(synth.normal_bf16((B, T, D), 900 + D))
    emb = _dev(synth.normal_bf16((B, 6 * D), 901, 0.1))
    sc, sh = emb[:, :D], emb[:, D:2 * D]
    w = _dev(synth.normal_bf16((D,), 902, 0.1, 1.0)) if weight else None
    ref = ops.rms_modulate(x, sc, sh, EPS, weight=w)
    stream = torch.cuda.current_stream().cuda_stream
    for call in range(2):
        y = torch.full_like(x, float("nan"))
        status = lib.dan_rms_modulate_noalloc(x.data_ptr(), None if w is None else w.data_ptr(),
                                              sc.data_ptr(), sh.data_ptr(), 6 * D, y.data_ptr(),
                                              B, T, D, EPS, stream)
        assert status == ops.DAN_OK, ops.status_string(status)
        torch.cuda.synchronize()
        assert torch.equal(y.view(torch.int16), ref.view(torch.int16)), f"call {call} differs"
    assert ops.device_status() == 0
