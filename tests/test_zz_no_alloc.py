"""dan_rms_modulate_noalloc through the C ABI.  It serves callers that cannot
allocate device memory (code inside a stream capture that forbids
allocation, or a runtime whose device memory belongs to its own caching
allocator); its scratch lives in a static device array that every call
shares and that keeps the previous call's contents.  So each case runs two
calls in a row and checks both against the CPU oracle bit for bit, and
against dan_rms_modulate.  Collected last, so that a run that stops at the
first failure has run every other test first."""
import numpy as np
import pytest
import torch

import oracle
from dit_adaln_norm_gb300 import build as dan_build
from dit_adaln_norm_gb300 import ops, synth

pytestmark = pytest.mark.gpu
EPS = 1e-6


def _dev(bits):
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16).cuda()


def _host(t):
    return t.contiguous().view(torch.int16).cpu().numpy().view(np.uint16)


# (B, T, D, weight): the eight- and twelve-warp shapes at 4096 (fewer and
# more than 24 rows per SM), 2048, and the team shapes of 6144 and 8192.
CASES = [(2, 1500, 4096, False), (1, 4216, 4096, False), (2, 1500, 2048, True),
         (1, 600, 6144, True), (1, 500, 8192, False)]


@pytest.mark.parametrize("B,T,D,weight", CASES)
def test_noalloc_matches_oracle_twice(B, T, D, weight):
    dan_build.build()
    oracle.build()
    lib = ops.load()
    x_h = synth.normal_bf16((B, T, D), 900 + D + T)
    emb_h = synth.normal_bf16((B, 6 * D), 901, 0.1)
    w_h = synth.normal_bf16((D,), 902, 0.1, 1.0) if weight else None
    x, emb = _dev(x_h), _dev(emb_h)
    sc, sh = emb[:, :D], emb[:, D:2 * D]
    w = _dev(w_h) if weight else None
    want = oracle.rms_modulate(x_h, emb_h[:, :D], emb_h[:, D:2 * D], EPS, weight=w_h)
    ref = _host(ops.rms_modulate(x, sc, sh, EPS, weight=w))
    assert np.array_equal(ref, want)
    stream = torch.cuda.current_stream().cuda_stream
    for call in range(2):
        y = torch.full_like(x, float("nan"))
        status = lib.dan_rms_modulate_noalloc(x.data_ptr(), None if w is None else w.data_ptr(),
                                              sc.data_ptr(), sh.data_ptr(), 6 * D, y.data_ptr(),
                                              B, T, D, EPS, stream)
        assert status == ops.DAN_OK, ops.status_string(status)
        torch.cuda.synchronize()
        assert np.array_equal(_host(y), want), f"call {call} differs from the oracle"
    assert ops.device_status() == 0
