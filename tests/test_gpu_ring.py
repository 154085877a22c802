"""The bulk-copy pipelines under stress, and their bounded waits.

Every kernel streams rows through shared-memory slots that each warp team
refills many times at these sizes; repeated launches must all be bit-exact
(a missing ordering between a warp's reads of a slot and its next refill
showed up as an occasional wrong row).  A wait that runs out must report
through the device status word and leave the context usable."""
import numpy as np
import pytest
import torch

import oracle
from dit_adaln_norm_gb300 import ops, synth
from _gpu import adaln, assert_bits_equal, from_dev, to_dev

pytestmark = pytest.mark.gpu
EPS = 1e-6
REPEATS = 12


def test_status_word_starts_clear():
    torch.cuda.synchronize()
    assert ops.device_status() == 0


def test_ln_ring_reuse_repeated():
    B, T, D = 1, 4096, 3072
    x = synth.outlier_rows_bf16((B, T, D), synth.SEED_X, synth.SEED_OUTLIER)
    (sc, sh), (dsc, dsh) = adaln(B, D, 2, synth.SEED_X + 1, 0.2)
    want = oracle.ln_modulate(x, sc, sh, EPS)
    xd = to_dev(x)
    for it in range(REPEATS):
        assert_bits_equal(from_dev(ops.ln_modulate(xd, dsc, dsh, EPS)), want, f"ln run {it}")
    torch.cuda.synchronize()
    assert ops.device_status() == 0


def test_rms_and_gated_ring_reuse_repeated():
    B, T, D = 1, 4216, 4096
    r = synth.normal_bf16((B, T, D), 700)
    h = synth.normal_bf16((B, T, D), 701)
    (g, sc, sh), (dg, dsc, dsh) = adaln(B, D, 3, 702, 0.1)
    want_y = oracle.rms_modulate(r, sc, sh, EPS)
    want_r, want_g = oracle.gated_rms_modulate(r, h, g, sc, sh, EPS)
    rd, hd = to_dev(r), to_dev(h)
    for it in range(REPEATS):
        assert_bits_equal(from_dev(ops.rms_modulate(rd, dsc, dsh, EPS)), want_y, f"rms run {it}")
        ro, yo = ops.gated_rms_modulate(rd, hd, dg, dsc, dsh, EPS)
        assert_bits_equal(from_dev(ro), want_r, f"gated r' run {it}")
        assert_bits_equal(from_dev(yo), want_g, f"gated y run {it}")
    torch.cuda.synchronize()
    assert ops.device_status() == 0


def test_qk_ring_reuse_repeated():
    H, Tt, Ti = 24, 256, 4096
    pt, pi = synth.packed_qkv(Tt, H, 710), synth.packed_qkv(Ti, H, 711)
    ws = synth.head_weights(4, 712)
    rt, ri = synth.rope_table(Tt), synth.rope_table(Ti, pos0=Tt)
    want = oracle.qk_norm_rope_epilogue(synth.split_qkv(pt, H), synth.split_qkv(pi, H), H, ws,
                                        rt, ri, EPS, EPS)
    args = (synth.split_qkv(to_dev(pt), H), synth.split_qkv(to_dev(pi), H),
            *[to_dev(w) for w in ws], torch.from_numpy(rt).cuda(), torch.from_numpy(ri).cuda(),
            EPS, EPS, H)
    for it in range(REPEATS // 2):
        for name, g, w in zip("qkv", ops.qk_norm_rope_epilogue(*args), want):
            assert_bits_equal(from_dev(g), w, f"qk {name} run {it}")
    torch.cuda.synchronize()
    assert ops.device_status() == 0


def test_wait_that_runs_out_reports_and_context_survives():
    """A wait on an mbarrier nothing completes gives up after 20 ms, records
    bit 1 and returns; the status read clears it; kernels still run."""
    torch.cuda.synchronize()
    assert ops.device_status() == 0
    ops.selftest_wait_timeout(20_000_000)
    torch.cuda.synchronize()
    assert ops.device_status() == 1
    assert ops.device_status() == 0
    B, T, D = 1, 300, 4096
    x = synth.normal_bf16((B, T, D), 720)
    (sc, sh), (dsc, dsh) = adaln(B, D, 2, 721, 0.1)
    assert_bits_equal(from_dev(ops.rms_modulate(to_dev(x), dsc, dsh, EPS)),
                      oracle.rms_modulate(x, sc, sh, EPS), "rms after the timeout test")
    torch.cuda.synchronize()
    assert ops.device_status() == 0
