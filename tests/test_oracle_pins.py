"""Pins of the CPU oracle to facts other than itself.

Each check below would fail under a plausible slip in the oracle: a wrong
rounding rule, a dropped term, a swapped loop order, a transposed operand or
a wrong pairing.  Sources: the closed forms of the adaLN norm+modulate target
(constant row and scale = -1 give y = shift; a +-a row gives +-1/sqrt(1+eps/a^2)),
the canonical order described in the "SGLang diffusion fused-op package
guide" (section "Norm + scale/shift (adaLN)"), hand-worked sums under
tests/golden/, and an fp64 brute force that must agree within 2 bf16 ULP
(y) and 1e-6 relative (fp32 rstd).
"""
import json
import os

import numpy as np
import pytest
import torch

from dit_adaln_norm_gb300 import synth

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")
EPS = 1e-6


# ------------------------------------------------------------------ helpers

def widen(bits):
    return (np.asarray(bits).astype(np.uint32) << 16).view(np.float32)


def bits_of(values_f32):
    return synth.to_bf16_bits(np.asarray(values_f32, np.float32))


def bf16_of_f64(v):
    """Round fp64 values to bf16 (through torch) and return them as fp64."""
    t = torch.from_numpy(np.asarray(v, np.float64)).to(torch.bfloat16).to(torch.float64)
    return t.numpy()


def bf16_ulp(mag):
    """Spacing of bf16 at magnitude |mag| (fp64), floored at the subnormal step."""
    mag = np.abs(np.asarray(mag, np.float64))
    _, e = np.frexp(np.where(mag > 0, mag, 1.0))
    return np.ldexp(1.0, np.maximum(e - 8, -133)) * np.where(mag > 0, 1.0, 0.0) + \
        np.where(mag > 0, 0.0, 2.0 ** -133)


def vec(B, D, values):
    return bits_of(np.broadcast_to(np.asarray(values, np.float32), (B, D)).copy())


# ----------------------------------------------------- c-0: bf16 rounding

def _reference_round(u32):
    """Independent formulation: nearest of the two bf16 neighbours in fp64,
    ties to the even bf16 pattern; values past the largest bf16 round to inf
    as if it were 2^128; NaN -> quiet NaN with its sign."""
    u32 = np.asarray(u32, np.uint32)
    lo = (u32 >> 16).astype(np.uint32)
    hi = lo + 1
    hi_is_inf = (hi & 0x7FFF) == 0x7F80
    with np.errstate(over="ignore", invalid="ignore"):
        f64 = u32.view(np.float32).astype(np.float64)
        lo_val = (lo << 16).view(np.float32).astype(np.float64)
        hi_val = np.where(hi_is_inf, np.copysign(2.0 ** 128, f64),
                          (hi << 16).astype(np.uint32).view(np.float32).astype(np.float64))
        d_lo = np.abs(f64 - lo_val)
        d_hi = np.abs(hi_val - f64)
    pick_hi = (d_hi < d_lo) | ((d_hi == d_lo) & (lo & 1 == 1))
    exact = (u32 & 0xFFFF) == 0
    out = np.where(pick_hi & ~exact, hi, lo).astype(np.uint16)
    nan = (u32 & 0x7FFFFFFF) > 0x7F800000
    return np.where(nan, ((u32 >> 16) & 0x8000) | 0x7FC0, out).astype(np.uint16)


def test_round_bf16_every_high_half_and_ties(orc):
    hi = np.arange(1 << 16, dtype=np.uint32) << 16
    lows = np.array([0x0000, 0x0001, 0x7FFF, 0x8000, 0x8001, 0xFFFF], np.uint32)
    u = (hi[:, None] | lows[None, :]).ravel()
    got = orc.round_bf16(u.view(np.float32))
    assert np.array_equal(got, _reference_round(u))


def test_round_bf16_random_words(orc):
    u = np.random.Generator(np.random.PCG64(7)).integers(0, 1 << 32, 2_000_000,
                                                          dtype=np.uint64).astype(np.uint32)
    assert np.array_equal(orc.round_bf16(u.view(np.float32)), _reference_round(u))


def test_round_bf16_matches_torch_cast_on_finite(orc):
    """torch's fp32 -> bf16 cast is a second, independent RNE implementation."""
    u = np.random.Generator(np.random.PCG64(8)).integers(0, 1 << 32, 500_000,
                                                          dtype=np.uint64).astype(np.uint32)
    f = u.view(np.float32)
    f = f[np.isfinite(f)]
    assert np.array_equal(orc.round_bf16(f), synth.to_bf16_bits(f))


# ---------------------------------------------- c-1: canonical RMS order

def _probe_row(p):
    D = p["D"]
    x = np.zeros(D, np.float32)
    cols = p["columns"]
    if "ones_thread" in cols:
        tpr = D // 64
        tx = cols["ones_thread"]
        for b in range(8):
            for v in range(8):
                x[8 * tpr * b + 8 * tx + v] = 1.0
    for c, val in cols["big"]:
        x[c] = val
    return x


@pytest.mark.parametrize("name", ["chain_v_fastest", "adjacent_pair_tree",
                                  "three_warps_padded_tree", "four_warps_tree",
                                  "non_power_of_two_width"])
def test_rms_order_probes(orc, name):
    probes = {p["name"]: p for p in json.load(open(os.path.join(GOLDEN,
                                                                "rms_order_probes.json")))["probes"]}
    p = probes[name]
    D = p["D"]
    x = bits_of(_probe_row(p))[None, None, :]
    zeros = vec(1, D, 0.0)
    _, st = orc.rms_modulate(x, zeros, zeros, p.get("eps", EPS), with_stats=True)
    assert st[0, 0] == np.float32(p["expected_s"]), (st[0, 0], p["expected_s"])
    if "expected_rstd" in p:
        assert st[0, 1] == np.float32(p["expected_rstd"]), (st[0, 1], p["expected_rstd"])


@pytest.mark.parametrize("D", [2048, 4096, 6144, 8192])
def test_rms_unit_magnitude_row(orc, D):
    """All +-1 (random signs): s = D exactly; with scale = shift = 0 and
    eps = 1e-6, y = +-1 exactly (1/sqrt(1 + 1e-6) rounds to 1 in bf16)."""
    sgn = np.where(np.random.Generator(np.random.PCG64(D)).random((3, D)) < 0.5, -1.0, 1.0)
    x = bits_of(sgn)[None]
    zeros = vec(1, D, 0.0)
    y, st = orc.rms_modulate(x, zeros, zeros, EPS, with_stats=True)
    assert np.all(st[:, 0] == D)
    assert np.array_equal(widen(y[0]), sgn.astype(np.float32))


@pytest.mark.parametrize("a", [0.5, 1.5, 3.0, 96.0, 2.0 ** -10])
def test_rms_alternating_closed_form(orc, a):
    """+-a row: y = +-1/sqrt(1 + eps/a^2) within one bf16 ULP; at a = 2^-10,
    a^2 is about eps, so eps moves y by a third."""
    D = 4096
    x = bits_of(a * (-1.0) ** np.arange(D))[None, None]
    zeros = vec(1, D, 0.0)
    y = orc.rms_modulate(x, zeros, zeros, EPS)
    expect = (-1.0) ** np.arange(D) / np.sqrt(1.0 + EPS / a ** 2)
    assert np.all(np.abs(widen(y[0, 0]) - expect) <= bf16_ulp(expect))


def test_scale_minus_one_gives_shift(orc):
    """o = bf(1 + (-1)) = 0, p = +-0, y = shift (as a value) for every variant."""
    B, T, D = 2, 5, 4096
    x = synth.normal_bf16((B, T, D), 3)
    shift = synth.normal_bf16((B, D), 4, 0.5)
    scale = vec(B, D, -1.0)
    for y in (orc.rms_modulate(x, scale, shift, EPS), orc.ln_modulate(x, scale, shift, EPS),
              orc.gated_rms_modulate(x, synth.normal_bf16((B, T, D), 5),
                                     synth.normal_bf16((B, D), 6, 0.1), scale, shift, EPS)[1]):
        assert np.array_equal(widen(y), np.broadcast_to(widen(shift)[:, None, :], (B, T, D)))


def test_zero_row_gives_shift(orc):
    B, T, D = 1, 2, 2048
    x = np.zeros((B, T, D), np.uint16)
    scale = synth.normal_bf16((B, D), 8, 0.3)
    shift = synth.normal_bf16((B, D), 9, 0.3)
    for y in (orc.rms_modulate(x, scale, shift, EPS), orc.ln_modulate(x, scale, shift, EPS)):
        assert np.array_equal(widen(y), np.broadcast_to(widen(shift)[:, None, :], (B, T, D)))


def test_rms_weight_one_and_two(orc):
    B, T, D = 1, 4, 4096
    x = synth.normal_bf16((B, T, D), 10)
    zeros = vec(B, D, 0.0)
    y0 = orc.rms_modulate(x, zeros, zeros, EPS)
    y1 = orc.rms_modulate(x, zeros, zeros, EPS, weight=bits_of(np.ones(D)))
    y2 = orc.rms_modulate(x, zeros, zeros, EPS, weight=bits_of(np.full(D, 2.0)))
    assert np.array_equal(y0, y1)
    assert np.array_equal(widen(y2), 2.0 * widen(y0))


def test_sign_flip_and_power_of_two_scaling(orc):
    """x -> -x negates n exactly; x -> 4x with eps = 0 leaves n unchanged
    (every operation scales exactly by a power of two)."""
    B, T, D = 1, 6, 3072
    x = synth.outlier_rows_bf16((B, T, D), 11, 12)
    zeros = vec(B, D, 0.0)
    neg = x ^ np.uint16(0x8000)
    x4 = bits_of(4.0 * widen(x))
    for fn, Dk in ((orc.ln_modulate, D), (orc.rms_modulate, 3072)):
        y = fn(x, zeros, zeros, EPS)
        assert np.array_equal(widen(fn(neg, zeros, zeros, EPS)), -widen(y))
        assert np.array_equal(fn(x4, zeros, zeros, 0.0), fn(x, zeros, zeros, 0.0))


# ------------------------------------------------- c-2: LayerNorm Welford

def test_ln_constant_rows(orc):
    B, T, D = 2, 7, 3072
    c = widen(synth.normal_bf16((B, T), 13, 3.0))
    x = bits_of(np.broadcast_to(c[..., None], (B, T, D)))
    scale = synth.normal_bf16((B, D), 14, 0.2)
    shift = synth.normal_bf16((B, D), 15, 0.2)
    y, st = orc.ln_modulate(x, scale, shift, EPS, with_stats=True)
    assert np.array_equal(st[:, 0], c.ravel()) and np.all(st[:, 1] == 0)
    assert np.array_equal(widen(y), np.broadcast_to(widen(shift)[:, None, :], (B, T, D)))


def test_ln_two_chain_combine_by_hand(orc):
    """D = 16: thread 0 holds eight 1s, thread 1 eight 3s.  Combine: n = 16,
    c = 8/16, delta = 2, mean = 1 + 2*0.5 = 2, m2 = 0 + 0 + (4*8)*0.5 = 16;
    var = 1, rstd = 1 (eps = 0), n = x - 2 = -+1."""
    x = bits_of(np.r_[np.ones(8), np.full(8, 3.0)])[None, None]
    zeros = vec(1, 16, 0.0)
    y, st = orc.ln_modulate(x, zeros, zeros, 0.0, with_stats=True)
    assert (st[0, 0], st[0, 1], st[0, 2]) == (2.0, 16.0, 1.0)
    assert np.array_equal(widen(y[0, 0]), np.r_[-np.ones(8), np.ones(8)].astype(np.float32))


def test_ln_three_chain_count_weights_by_hand(orc):
    """D = 24: threads 0,1,2 hold eight 1s, 5s, 3s.  shfl.down order pairs
    (t0 + t2) first: n 16, mean 2, m2 (2*2*8)*0.5 = 16; then + t1 (n 8,
    mean 5): c = rn(8/24), delta = 3, mean = 2 + rn(3*c) = 3 and
    m2 = 16 + rn(rn(9*16)*c) = 64, all exact after rounding.  Weighting by
    nA/n instead of nB/n would give mean 4."""
    x = bits_of(np.r_[np.ones(8), np.full(8, 5.0), np.full(8, 3.0)])[None, None]
    zeros = vec(1, 24, 0.0)
    _, st = orc.ln_modulate(x, zeros, zeros, 0.0, with_stats=True)
    assert (st[0, 0], st[0, 1]) == (3.0, 64.0)


@pytest.mark.parametrize("a", [1.0, 0.25, 3.0, 2.0 ** -10])
def test_ln_alternating_closed_form(orc, a):
    """+-a alternating row: mean 0, var a^2, y = +-1/sqrt(1 + eps/a^2)
    within 2 bf16 ULP (Welford rounds from n = 3 on); at a = 2^-10 the eps
    term is as large as the variance."""
    D = 3072
    sgn = (-1.0) ** np.arange(D)
    x = bits_of(a * sgn)[None, None]
    zeros = vec(1, D, 0.0)
    y = orc.ln_modulate(x, zeros, zeros, EPS)
    expect = sgn / np.sqrt(1.0 + EPS / a ** 2)
    assert np.all(np.abs(widen(y[0, 0]) - expect) <= 2 * bf16_ulp(expect))


# ----------------------------------------------------- c-6: fp64 brute force

def _check_modulated(y, n64, scale, shift):
    """y (oracle bits) against the fp64 normalised value n64 carried through
    the bf16 modulate boundaries: within 2 bf16 ULP of max(|p|, |shift|)."""
    o = widen(bits_of(1.0 + widen(scale).astype(np.float32))).astype(np.float64)
    p = bf16_of_f64(bf16_of_f64(n64) * o)
    sh = widen(shift).astype(np.float64)
    y64 = bf16_of_f64(p + sh)
    tol = 2 * bf16_ulp(np.maximum(np.abs(p), np.abs(sh)))
    err = np.abs(widen(y).astype(np.float64) - y64)
    assert np.all(err <= tol), float((err / tol).max())


@pytest.mark.parametrize("D", [64, 128, 256, 2048, 4096])
def test_rms_fp64_brute_force(orc, D):
    B, T = 2, 24
    x = synth.normal_bf16((B, T, D), 20 + D)
    scale, shift = synth.adaln_vectors(B, D, 2, 21, 0.1)
    y, st = orc.rms_modulate(x, scale, shift, EPS, with_stats=True)
    xf = widen(x).astype(np.float64)
    s64 = (xf ** 2).sum(-1)
    rstd64 = 1.0 / np.sqrt(s64 / D + EPS)
    assert np.all(np.abs(st[:, 1] / rstd64.ravel() - 1.0) <= 1e-6)
    assert np.all(np.abs(st[:, 0] / s64.ravel() - 1.0) <= 1e-5)
    _check_modulated(y, xf * rstd64[..., None], scale[:, None, :], shift[:, None, :])


def test_gated_fp64_brute_force(orc):
    B, T, D = 1, 16, 4096
    r = synth.normal_bf16((B, T, D), 30)
    h = synth.normal_bf16((B, T, D), 31)
    gate, scale, shift = synth.adaln_vectors(B, D, 3, 32, 0.1)
    r_out, y = orc.gated_rms_modulate(r, h, gate, scale, shift, EPS)
    exact = widen(r).astype(np.float64) + widen(gate)[:, None, :].astype(np.float64) * \
        widen(h).astype(np.float64)
    gh = np.abs(widen(gate)[:, None, :].astype(np.float64) * widen(h))
    mag = np.maximum(np.maximum(np.abs(widen(r)), gh), np.abs(widen(r_out)))
    assert np.all(np.abs(widen(r_out) - exact) <= bf16_ulp(mag))
    # y is the RMS+modulate of r' (same oracle, consistency)...
    assert np.array_equal(y, orc.rms_modulate(r_out, scale, shift, EPS))
    # ...and within tolerance of the fp64 chain on r'.
    rf = widen(r_out).astype(np.float64)
    rstd64 = 1.0 / np.sqrt((rf ** 2).mean(-1) + EPS)
    _check_modulated(y, rf * rstd64[..., None], scale[:, None, :], shift[:, None, :])


def test_gated_special_gates(orc):
    """gate = 0 -> r' = r; gate = 1 -> r' = bf16 of the exact r + h."""
    B, T, D = 1, 3, 2048
    r = synth.normal_bf16((B, T, D), 33)
    h = synth.normal_bf16((B, T, D), 34)
    zeros = vec(B, D, 0.0)
    r0, _ = orc.gated_rms_modulate(r, h, zeros, zeros, zeros, EPS)
    assert np.array_equal(widen(r0), widen(r))
    r1, _ = orc.gated_rms_modulate(r, h, vec(B, D, 1.0), zeros, zeros, EPS)
    exact = widen(r).astype(np.float64) + widen(h).astype(np.float64)
    assert np.array_equal(widen(r1), bf16_of_f64(exact).astype(np.float32))


@pytest.mark.parametrize("D,outliers", [(8, False), (64, False), (1040, False),
                                        (3072, True), (4096, False), (4096, True)])
def test_ln_fp64_brute_force(orc, D, outliers):
    B, T = 2, 24
    x = (synth.outlier_rows_bf16((B, T, D), 40 + D, 2) if outliers
         else synth.normal_bf16((B, T, D), 40 + D))
    scale, shift = synth.adaln_vectors(B, D, 2, 41, 0.2)
    y, st = orc.ln_modulate(x, scale, shift, EPS, with_stats=True)
    xf = widen(x).astype(np.float64)
    mean64 = xf.mean(-1)
    var64 = ((xf - mean64[..., None]) ** 2).mean(-1)
    rstd64 = 1.0 / np.sqrt(var64 + EPS)
    assert np.all(np.abs(st[:, 2] / rstd64.ravel() - 1.0) <= 1e-6)
    assert np.all(np.abs(st[:, 0] - mean64.ravel()) <= 1e-6 * np.sqrt(var64.ravel()))
    _check_modulated(y, (xf - mean64[..., None]) * rstd64[..., None],
                     scale[:, None, :], shift[:, None, :])


def test_batch_stride_and_batching_consistency(orc):
    """A [B, D] strided view gives each batch's rows its own vectors: the same
    as running every batch alone with contiguous vectors."""
    B, T, D = 3, 5, 4096
    x = synth.normal_bf16((B, T, D), 50)
    scale, shift = synth.adaln_vectors(B, D, 2, 51, 0.2, chunks=6)
    assert scale.strides[0] == 6 * D * 2
    for fn in (orc.rms_modulate, orc.ln_modulate):
        y = fn(x, scale, shift, EPS)
        for b in range(B):
            yb = fn(x[b:b + 1], np.ascontiguousarray(scale[b:b + 1]),
                    np.ascontiguousarray(shift[b:b + 1]), EPS)
            assert np.array_equal(y[b:b + 1], yb)


# -------------------------------------------- c-5: QK norm + RoPE epilogue

def _qk_inputs(Tt, Ti, H, seed):
    pt = synth.packed_qkv(Tt, H, seed)
    pi = synth.packed_qkv(Ti, H, seed + 1)
    ws = synth.head_weights(4, seed + 2)
    return pt, pi, ws


def _rope_const(T, c, s):
    return np.concatenate([np.full((T, 64), c, np.float32), np.full((T, 64), s, np.float32)], 1)


def test_qk_identity_and_quarter_turn(orc):
    """cos = 1, sin = 0 leaves the normalised head unchanged; cos = 0,
    sin = 1 maps the interleaved pair (a, b) to (-b, a) exactly."""
    Tt, Ti, H = 3, 5, 4
    pt, pi, ws = _qk_inputs(Tt, Ti, H, 60)
    txt, img = synth.split_qkv(pt, H), synth.split_qkv(pi, H)
    q1, k1, v1 = orc.qk_norm_rope_epilogue(txt, img, H, ws, _rope_const(Tt, 1, 0),
                                           _rope_const(Ti, 1, 0), EPS, EPS)
    q2, k2, v2 = orc.qk_norm_rope_epilogue(txt, img, H, ws, _rope_const(Tt, 0, 1),
                                           _rope_const(Ti, 0, 1), EPS, EPS)
    for n, r in ((q1, q2), (k1, k2)):
        nf, rf = widen(n), widen(r)
        assert np.array_equal(rf[..., 0::2], -nf[..., 1::2])
        assert np.array_equal(rf[..., 1::2], nf[..., 0::2])
    assert np.array_equal(v1, v2)


def test_qk_unit_head_closed_form(orc):
    """A head of +-1 with weight 1 and cos = 1, sin = 0 comes out as +-1."""
    Tt, Ti, H = 2, 2, 3
    sgn = np.where(np.random.Generator(np.random.PCG64(61)).random((Tt + Ti, 3 * H * 128)) < 0.5,
                   -1.0, 1.0)
    packed = bits_of(sgn)
    ones = [bits_of(np.ones(128))] * 4
    q, k, v = orc.qk_norm_rope_epilogue(synth.split_qkv(packed[:Tt], H),
                                        synth.split_qkv(packed[Tt:], H), H, ones,
                                        _rope_const(Tt, 1, 0), _rope_const(Ti, 1, 0), EPS, EPS)
    W = H * 128
    assert np.array_equal(widen(q).reshape(-1, W), sgn[:, :W].astype(np.float32))
    assert np.array_equal(widen(k).reshape(-1, W), sgn[:, W:2 * W].astype(np.float32))


def test_qk_small_head_eps_per_stream(orc):
    """A head of +-a with a = 2^-10 (a^2 about eps), weight 1, cos = 1 and
    sin = 0: q = k = +-1/sqrt(1 + eps_s/a^2) within one bf16 ULP, with the
    text stream's eps for text tokens and the image stream's for image
    tokens (the epilogue passes each stream's norm epsilon)."""
    Tt, Ti, H, a = 2, 3, 2, 2.0 ** -10
    eps_t, eps_i = 1e-6, 4e-6
    sgn = np.where(np.random.Generator(np.random.PCG64(62)).random((Tt + Ti, 3 * H * 128)) < 0.5,
                   -1.0, 1.0)
    packed = bits_of(a * sgn)
    ones = [bits_of(np.ones(128))] * 4
    q, k, _ = orc.qk_norm_rope_epilogue(synth.split_qkv(packed[:Tt], H),
                                        synth.split_qkv(packed[Tt:], H), H, ones,
                                        _rope_const(Tt, 1, 0), _rope_const(Ti, 1, 0), eps_t, eps_i)
    W = H * 128
    mag = np.r_[np.full(Tt, 1.0 / np.sqrt(1.0 + eps_t / a ** 2)),
                np.full(Ti, 1.0 / np.sqrt(1.0 + eps_i / a ** 2))][:, None]
    for out, cols in ((q, slice(0, W)), (k, slice(W, 2 * W))):
        expect = sgn[:, cols] * mag
        err = np.abs(widen(out).reshape(-1, W) - expect)
        assert np.all(err <= bf16_ulp(expect))


def test_qk_v_copy_and_joint_order(orc):
    Tt, Ti, H = 4, 6, 2
    pt, pi, ws = _qk_inputs(Tt, Ti, H, 62)
    txt, img = synth.split_qkv(pt, H), synth.split_qkv(pi, H)
    _, _, v = orc.qk_norm_rope_epilogue(txt, img, H, ws, synth.rope_table(Tt),
                                        synth.rope_table(Ti), EPS, EPS)
    assert np.array_equal(v[:Tt].reshape(Tt, -1), txt[2])
    assert np.array_equal(v[Tt:].reshape(Ti, -1), img[2])


def test_qk_fp64_brute_force(orc):
    Tt, Ti, H = 8, 24, 3
    pt, pi, ws = _qk_inputs(Tt, Ti, H, 63)
    txt, img = synth.split_qkv(pt, H), synth.split_qkv(pi, H)
    rt, ri = synth.rope_table(Tt), synth.rope_table(Ti, pos0=17)
    eps_t, eps_i = 1e-6, 1e-5
    q, k, v, rs = orc.qk_norm_rope_epilogue(txt, img, H, ws, rt, ri, eps_t, eps_i,
                                            with_stats=True)
    for s, (src, rope, eps, wq, wk, row0) in enumerate(
            ((txt, rt, eps_t, ws[0], ws[1], 0), (img, ri, eps_i, ws[2], ws[3], Tt))):
        T = src[0].shape[0]
        for which, (x, w, out) in enumerate(((src[0], wq, q), (src[1], wk, k))):
            xf = widen(x).astype(np.float64).reshape(T, H, 128)
            rstd64 = 1.0 / np.sqrt((xf ** 2).mean(-1) + eps)
            got_rstd = rs[row0:row0 + T, which, :]
            assert np.all(np.abs(got_rstd / rstd64 - 1.0) <= 1e-6)
            n = bf16_of_f64(xf * rstd64[..., None] * widen(w).astype(np.float64))
            a, b = n[..., 0::2], n[..., 1::2]
            c = rope[:, None, :64].astype(np.float64)
            sn = rope[:, None, 64:].astype(np.float64)
            e0, e1 = a * c - b * sn, a * sn + b * c
            tol = 2 * bf16_ulp(np.maximum(np.abs(a), np.abs(b)))
            o = widen(out[row0:row0 + T]).astype(np.float64)
            assert np.all(np.abs(o[..., 0::2] - e0) <= tol)
            assert np.all(np.abs(o[..., 1::2] - e1) <= tol)


# ------------------------------------- hand-worked probes under tests/golden

def _golden(name):
    return {p["name"]: p for p in json.load(open(os.path.join(GOLDEN, name)))["probes"]}


def _runs(runs):
    return np.concatenate([np.full(n, v, np.float64) for v, n in runs])


@pytest.mark.parametrize("name", ["welford_reciprocal", "lane_tree_down_order", "cross_warp_order",
                                  "combine_m2_product_order", "cross_warp_operand_order"])
def test_ln_order_probes(orc, name):
    p = _golden("ln_order_probes.json")[name]
    xs = np.asarray(p["x"], np.float64) if "x" in p else _runs(p["x_runs"])
    D = p["D"]
    assert xs.size == D
    zeros = vec(1, D, 0.0)
    _, st = orc.ln_modulate(bits_of(xs)[None, None], zeros, zeros, p["eps"], with_stats=True)
    assert st[0, 0] == np.float32(p["expected_mean"]), (float(st[0, 0]), p["expected_mean"])
    if "expected_m2" in p:
        assert st[0, 1] == np.float32(p["expected_m2"]), (float(st[0, 1]), p["expected_m2"])


def test_one_plus_scale_tie_probe(orc):
    B, T, D = 1, 4, 4096
    x = synth.normal_bf16((B, T, D), 70)
    shift = synth.normal_bf16((B, D), 71, 0.2)
    for fn in (orc.rms_modulate, orc.ln_modulate):
        assert np.array_equal(fn(x, vec(B, D, 2.0 ** -8), shift, EPS),
                              fn(x, vec(B, D, 0.0), shift, EPS))
        assert np.array_equal(fn(x, vec(B, D, 3 * 2.0 ** -8), shift, EPS),
                              fn(x, vec(B, D, 2.0 ** -6), shift, EPS))


def test_rms_product_probe(orc):
    p = _golden("rounding_boundary_probes.json")["rms_product_rounded_before_shift"]
    D = p["D"]
    y = orc.rms_modulate(bits_of(np.full((1, 1, D), p["x"])), vec(1, D, p["scale"]),
                         vec(1, D, p["shift"]), p["eps"], weight=bits_of(np.full(D, p["weight"])))
    assert np.all(widen(y) == np.float32(p["expected_y"]))


def test_ln_product_probe(orc):
    p = _golden("rounding_boundary_probes.json")["ln_product_rounded_before_shift"]
    D = p["D"]
    y = orc.ln_modulate(bits_of(_runs(p["x_runs"]))[None, None], vec(1, D, p["scale"]),
                        vec(1, D, p["shift"]), p["eps"])
    expect = _runs([(v, n) for v, (_, n) in zip(p["expected_y_runs"], p["x_runs"])])
    assert np.array_equal(widen(y[0, 0]), expect.astype(np.float32))


def test_gated_product_probe(orc):
    p = _golden("rounding_boundary_probes.json")["gated_product_rounded_before_add"]
    D = p["D"]
    r_out, _ = orc.gated_rms_modulate(bits_of(np.full((1, 1, D), p["r"])),
                                      bits_of(np.full((1, 1, D), p["h"])), vec(1, D, p["gate"]),
                                      vec(1, D, 0.0), vec(1, D, 0.0), EPS)
    assert np.all(widen(r_out) == np.float32(p["expected_r_out"]))


def test_weight_single_rounding_probe(orc):
    p = _golden("rounding_boundary_probes.json")["weight_single_rounding"]
    D = p["D"]
    x = np.tile(np.asarray(p["x_alternating"], np.float64), D // 2)
    y = orc.rms_modulate(bits_of(x)[None, None], vec(1, D, p["scale"]), vec(1, D, p["shift"]),
                         p["eps"], weight=bits_of(np.full(D, p["weight"])))
    expect = np.tile(np.asarray(p["expected_y_alternating"], np.float32), D // 2)
    assert np.array_equal(widen(y[0, 0]), expect)


def test_rms_weight_product_order_probe(orc):
    """rn(rn(x*rstd)*w): rstd multiplies first, then the weight (ERNIE's
    (bf16)(x*rstd*w) read left to right); rn(x*w)*rstd lands one fp32 ulp
    below a bf16 midpoint and rounds the other way."""
    p = _golden("rounding_boundary_probes.json")["rms_weight_product_order"]
    D = p["D"]
    x = np.tile(np.asarray(p["x_alternating"], np.float64), D // 2)
    y = orc.rms_modulate(bits_of(x)[None, None], vec(1, D, p["scale"]), vec(1, D, p["shift"]),
                         p["eps"], weight=bits_of(np.full(D, p["weight"])))
    expect = np.tile(np.asarray(p["expected_y_alternating"], np.float32), D // 2)
    assert np.array_equal(widen(y[0, 0]), expect)


def test_qk_weight_product_order_probe(orc):
    """Per-head norm with weight: rn(rn(x*rstd)*w), not x*rn(rstd*w)."""
    p = _golden("rounding_boundary_probes.json")["qk_weight_product_order"]
    hd, H = p["head_dim"], 2
    head = np.tile(np.asarray(p["x_alternating"], np.float32), hd // 2)
    row = np.tile(head, 3 * H)
    packed = bits_of(np.stack([row, row]))
    ws = [bits_of(np.full(hd, p["weight"]))] * 4
    rope = _rope_const_hd(1, hd, p["cos"], p["sin"])
    q, k, v = orc.qk_norm_rope_epilogue(
        synth.split_qkv(packed[:1], H, hd), synth.split_qkv(packed[1:], H, hd), H, ws, rope,
        rope, p["eps"], p["eps"], head_dim=hd)
    expect = np.tile(np.asarray(p["expected_alternating"], np.float32), hd // 2)
    for out in (q, k):
        assert np.array_equal(widen(out).reshape(-1, hd), np.broadcast_to(expect, (2 * H, hd)))
    assert np.array_equal(v.reshape(2, -1), packed[:, 2 * H * hd:])


def test_ln_combine_count_weighting_probe(orc):
    """The combine's m2 term is rn(rn(rn(delta^2)*nA)*rn(nB/n)) (A the lower
    state): at counts 24 and 16 the other weighting changes m2 by one ulp,
    and at this eps the x = 2 outputs by one bf16 step."""
    p = _golden("ln_order_probes.json")["combine_count_weighting"]
    D = p["D"]
    xs = _runs(p["x_runs"])
    zeros = vec(1, D, 0.0)
    y, st = orc.ln_modulate(bits_of(xs)[None, None], zeros, zeros, p["eps"], with_stats=True)
    assert st[0, 0] == np.float32(p["expected_mean"]), float(st[0, 0])
    assert st[0, 1] == np.float32(p["expected_m2"]), float(st[0, 1])
    expect = _runs([(v, n) for v, (_, n) in zip(p["expected_y_runs"], p["x_runs"])])
    assert np.array_equal(widen(y[0, 0]), expect.astype(np.float32))


# ------------------------------------- LayerNorm + modulate + static FP8

def e4m3_decode(code):
    """Value of an E4M3 ("e4m3fn") code from the format's definition: sign,
    4 exponent bits (bias 7), 3 mantissa bits, subnormals at exponent 0,
    S.1111.111 is NaN.  Written independently of the oracle's encoder."""
    code = int(code)
    s = -1.0 if code & 0x80 else 1.0
    e, m = (code >> 3) & 0xF, code & 7
    if e == 15 and m == 7:
        return float("nan")
    if e == 0:
        return s * (m / 8.0) * 2.0 ** -6
    return s * (1.0 + m / 8.0) * 2.0 ** (e - 7)


FINITE_CODES = [c for c in range(256) if (c & 0x7F) != 0x7F]


def test_e4m3_decoder_matches_torch():
    # the test's own decoder agrees with torch's float8_e4m3fn on every code
    t = torch.tensor(list(range(256)), dtype=torch.uint8).view(torch.float8_e4m3fn).float().numpy()
    for c in range(256):
        want = e4m3_decode(c)
        assert (np.isnan(want) and np.isnan(t[c])) or want == t[c], c


def test_e4m3_every_finite_code_round_trips(orc):
    vals = np.array([e4m3_decode(c) for c in FINITE_CODES], np.float32)
    got = orc.fp8_e4m3(vals)
    assert list(got) == FINITE_CODES
    assert int(got[FINITE_CODES.index(0x7E)]) == 0x7E and e4m3_decode(0x7E) == 448.0


def test_e4m3_midpoints_round_to_even_code(orc):
    pos = sorted((e4m3_decode(c), c) for c in range(0x7F))  # +0 .. 448
    mids, want = [], []
    for (a, ca), (b, cb) in zip(pos, pos[1:]):
        mids.append((a + b) / 2)                      # exact in fp32
        want.append(ca if ca % 2 == 0 else cb)        # ties to the even mantissa
    got = orc.fp8_e4m3(np.array(mids, np.float32))
    assert list(got) == want
    assert list(orc.fp8_e4m3(-np.array(mids, np.float32))) == [w | 0x80 for w in want]


def test_e4m3_saturation_and_specials(orc):
    v = np.array([448.0, 449.0, 463.9, 464.0, 480.0, 1e30, np.inf, -500.0, -np.inf,
                  np.nan, 0.0, -0.0, 2.0 ** -10, 2.0 ** -9, 2.0 ** -6 - 2.0 ** -10], np.float32)
    got = [int(c) for c in orc.fp8_e4m3(v)]
    assert got[:9] == [0x7E] * 7 + [0xFE, 0xFE]
    assert got[9] == 0x7F and got[10] == 0x00 and got[11] == 0x80
    assert got[12] == 0x00            # half the smallest subnormal: tie to even (zero)
    assert got[13] == 0x01            # the smallest subnormal
    assert got[14] == 0x08            # 2^-6 - 2^-10 is the midpoint 7.5/8: rounds to even 8/8


def test_e4m3_matches_torch_cast_in_range(orc):
    rng = np.random.default_rng(21)
    v = np.concatenate([rng.normal(0, 1, 20000), rng.normal(0, 100, 20000),
                        rng.uniform(-447, 447, 20000), rng.normal(0, 2.0 ** -7, 20000)])
    v = v.astype(np.float32)
    want = torch.from_numpy(v).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(orc.fp8_e4m3(v), want)


def test_e4m3_brute_force_nearest(orc):
    rng = np.random.default_rng(22)
    v = (rng.normal(0, 30, 3000) * rng.choice([1.0, 2.0 ** -8], 3000)).astype(np.float32)
    vals = np.array([e4m3_decode(c) for c in FINITE_CODES])
    got = orc.fp8_e4m3(v)
    for x, g in zip(v.astype(np.float64), got):
        d = np.abs(vals - min(max(x, -448.0), 448.0))
        best = [FINITE_CODES[i] for i in np.flatnonzero(d == d.min())]
        best = [c for c in best if (c & 0x80) == (0x80 if np.signbit(x) else 0)] or best
        want = min(best, key=lambda c: (c & 1, c))  # a tie goes to the even mantissa
        assert int(g) == want, (x, int(g), want)


def test_ln_fp8_constant_rows_quantise_shift(orc):
    B, T, D = 2, 5, 3072
    c = widen(synth.normal_bf16((B, T), 31, 2.0))
    x = bits_of(np.broadcast_to(c[..., None], (B, T, D)))
    scale = synth.normal_bf16((B, D), 32, 0.2)
    shift = synth.normal_bf16((B, D), 33, 3.0)
    qscale = 0.0625  # 1/qscale = 16 exactly
    q = orc.ln_modulate_fp8(x, scale, shift, qscale, EPS)
    want = torch.from_numpy(widen(shift) * np.float32(16.0)).to(torch.float8_e4m3fn)
    want = want.view(torch.uint8).numpy()
    assert np.array_equal(q, np.broadcast_to(want[:, None, :], (B, T, D)))


def test_ln_fp8_is_quantised_ln_modulate(orc):
    x = synth.outlier_rows_bf16((1, 64, 4096), 34, synth.SEED_OUTLIER)
    scale = synth.normal_bf16((1, 4096), 35, 0.2)
    shift = synth.normal_bf16((1, 4096), 36, 0.2)
    for qscale in (1.0, 0.02, 3.0):
        inv = np.float32(1.0) / np.float32(qscale)
        y = orc.ln_modulate(x, scale, shift, EPS)
        want = torch.from_numpy(widen(y) * inv).clamp(-448, 448).to(torch.float8_e4m3fn)
        assert np.array_equal(orc.ln_modulate_fp8(x, scale, shift, qscale, EPS),
                              want.view(torch.uint8).numpy())


def test_ln_fp8_scale_applied_as_reciprocal_multiply(orc):
    """The static scale is applied as rn(y * rn(1/qscale)), the reading the
    FP8 producer is built on, not as rn(y / qscale): at qscale = 7 the two
    round to different E4M3 codes for some bf16 y.  Constant rows make y
    equal to shift exactly (scale = 0, so bf16(1 + scale) = 1)."""
    bits = np.arange(0x0001, 0x7F80, dtype=np.uint32)
    yv = (bits << 16).view(np.float32)
    yv = yv[yv < 448.0 * 7.0]
    qs = np.float32(7.0)
    mul = torch.from_numpy(yv * (np.float32(1.0) / qs)).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    div = torch.from_numpy(yv / qs).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    split = yv[mul != div]
    assert split.size > 0  # the two readings differ somewhere
    D = 8 * ((split.size + 7) // 8)
    shift = np.zeros((1, D), np.float32)
    shift[0, :split.size] = split
    shift_bits = bits_of(shift)
    x = bits_of(np.full((1, 3, D), 1.5, np.float32))
    scale = bits_of(np.zeros((1, D), np.float32))
    q = orc.ln_modulate_fp8(x, scale, shift_bits, 7.0, EPS)
    want = torch.from_numpy(widen(shift_bits) * (np.float32(1.0) / qs)).to(torch.float8_e4m3fn)
    assert np.array_equal(q, np.broadcast_to(want.view(torch.uint8).numpy()[:, None, :], (1, 3, D)))
    assert not np.array_equal(q[0, 0, :split.size], div[mul != div])


# ---------------------------------------------- gated residual + LayerNorm

def test_gated_ln_residual_and_composition(orc):
    B, T, D = 2, 9, 3072
    r = synth.normal_bf16((B, T, D), 40)
    h = synth.normal_bf16((B, T, D), 41)
    gate, scale, shift = synth.adaln_vectors(B, D, 3, 42, 0.1)
    r_out, y = orc.gated_ln_modulate(r, h, gate, scale, shift, EPS)
    # r' independently: round(gate*h) then round(r + that), in torch bf16 ops
    tg = torch.from_numpy(widen(gate)[:, None, :]).to(torch.bfloat16)
    th = torch.from_numpy(widen(h)).to(torch.bfloat16)
    tr = torch.from_numpy(widen(r)).to(torch.bfloat16)
    want_r = (tr + tg * th).float().numpy()
    assert np.array_equal(widen(r_out), want_r)
    # y is the LayerNorm + modulate of r'
    assert np.array_equal(y, orc.ln_modulate(r_out, scale, shift, EPS))


def test_gated_ln_zero_gate_is_ln_of_residual(orc):
    B, T, D = 1, 5, 1040
    r = synth.outlier_rows_bf16((B, T, D), 43, synth.SEED_OUTLIER)
    h = synth.normal_bf16((B, T, D), 44)
    zeros = vec(B, D, 0.0)
    scale = synth.normal_bf16((B, D), 45, 0.2)
    shift = synth.normal_bf16((B, D), 46, 0.2)
    r_out, y = orc.gated_ln_modulate(r, h, zeros, scale, shift, EPS)
    assert np.array_equal(r_out, r)
    assert np.array_equal(y, orc.ln_modulate(r, scale, shift, EPS))


# ------------------------------- QK epilogue: head_dim 64 and neox rotation

def _rope_const_hd(T, hd, c, s):
    return np.concatenate([np.full((T, hd // 2), c, np.float32),
                           np.full((T, hd // 2), s, np.float32)], 1)


@pytest.mark.parametrize("hd", [64, 128])
def test_qk_neox_identity_and_quarter_turn(orc, hd):
    """neox: cos = 1, sin = 0 leaves the normalised head as the interleaved
    identity does; cos = 0, sin = 1 maps (x_i, x_{i+h}) to (-x_{i+h}, x_i)."""
    Tt, Ti, H = 3, 4, 3
    pt, pi = synth.packed_qkv(Tt, H, 70, hd), synth.packed_qkv(Ti, H, 71, hd)
    ws = synth.head_weights(4, 72, hd)
    txt, img = synth.split_qkv(pt, H, hd), synth.split_qkv(pi, H, hd)
    run = lambda c, s, neox: orc.qk_norm_rope_epilogue(
        txt, img, H, ws, _rope_const_hd(Tt, hd, c, s), _rope_const_hd(Ti, hd, c, s), EPS, EPS,
        head_dim=hd, neox=neox)
    q_id, k_id, _ = run(1, 0, False)
    q1, k1, v1 = run(1, 0, True)
    q2, k2, v2 = run(0, 1, True)
    assert np.array_equal(q1, q_id) and np.array_equal(k1, k_id)
    h = hd // 2
    for n, r in ((q1, q2), (k1, k2)):
        nf, rf = widen(n), widen(r)
        assert np.array_equal(rf[..., :h], -nf[..., h:])
        assert np.array_equal(rf[..., h:], nf[..., :h])
    assert np.array_equal(v1, v2) and np.array_equal(v1.reshape(Tt + Ti, -1)[:Tt], txt[2])


def test_qk_head_dim_64_unit_head(orc):
    Tt, Ti, H, hd = 2, 3, 5, 64
    sgn = np.where(np.random.Generator(np.random.PCG64(73)).random((Tt + Ti, 3 * H * hd)) < 0.5,
                   -1.0, 1.0)
    packed = bits_of(sgn)
    ones = [bits_of(np.ones(hd))] * 4
    q, k, _ = orc.qk_norm_rope_epilogue(synth.split_qkv(packed[:Tt], H, hd),
                                        synth.split_qkv(packed[Tt:], H, hd), H, ones,
                                        _rope_const_hd(Tt, hd, 1, 0),
                                        _rope_const_hd(Ti, hd, 1, 0), EPS, EPS, head_dim=hd)
    W = H * hd
    assert np.array_equal(widen(q).reshape(-1, W), sgn[:, :W].astype(np.float32))
    assert np.array_equal(widen(k).reshape(-1, W), sgn[:, W:2 * W].astype(np.float32))


@pytest.mark.parametrize("hd,neox", [(64, False), (64, True), (128, True)])
def test_qk_variants_fp64_brute_force(orc, hd, neox):
    Tt, Ti, H = 6, 20, 3
    pt, pi = synth.packed_qkv(Tt, H, 74, hd), synth.packed_qkv(Ti, H, 75, hd)
    ws = synth.head_weights(4, 76, hd)
    txt, img = synth.split_qkv(pt, H, hd), synth.split_qkv(pi, H, hd)
    rt, ri = synth.rope_table(Tt, hd), synth.rope_table(Ti, hd, pos0=11)
    q, k, _, rs = orc.qk_norm_rope_epilogue(txt, img, H, ws, rt, ri, EPS, EPS, with_stats=True,
                                            head_dim=hd, neox=neox)
    h = hd // 2
    for src, rope, wq, wk, row0 in ((txt, rt, ws[0], ws[1], 0), (img, ri, ws[2], ws[3], Tt)):
        T = src[0].shape[0]
        for which, (x, w, out) in enumerate(((src[0], wq, q), (src[1], wk, k))):
            xf = widen(x).astype(np.float64).reshape(T, H, hd)
            rstd64 = 1.0 / np.sqrt((xf ** 2).mean(-1) + EPS)
            assert np.all(np.abs(rs[row0:row0 + T, which, :] / rstd64 - 1.0) <= 1e-6)
            n = bf16_of_f64(xf * rstd64[..., None] * widen(w).astype(np.float64))
            a, b = (n[..., :h], n[..., h:]) if neox else (n[..., 0::2], n[..., 1::2])
            c = rope[:, None, :h].astype(np.float64)
            sn = rope[:, None, h:].astype(np.float64)
            e0, e1 = a * c - b * sn, a * sn + b * c
            tol = 2 * bf16_ulp(np.maximum(np.abs(a), np.abs(b)))
            o = widen(out[row0:row0 + T]).astype(np.float64)
            o0, o1 = (o[..., :h], o[..., h:]) if neox else (o[..., 0::2], o[..., 1::2])
            assert np.all(np.abs(o0 - e0) <= tol) and np.all(np.abs(o1 - e1) <= tol)


# ---------------------------------- residual gating in the transposed layout

def test_gated_residual_transposed_against_torch(orc):
    B, D, T = 2, 72, 37
    r = synth.normal_bf16((B, D, T), 80)
    h = synth.normal_bf16((B, T, D), 81)
    gate = synth.normal_bf16((B, D), 82, 0.5)
    got = orc.gated_residual_transposed(r, h, gate)
    tr = torch.from_numpy(widen(r)).to(torch.bfloat16)
    th = torch.from_numpy(widen(h)).to(torch.bfloat16).transpose(1, 2)   # logical [B, D, T]
    tg = torch.from_numpy(widen(gate)).to(torch.bfloat16)[:, :, None]
    want = (tr + tg * th).float().numpy()
    assert np.array_equal(widen(got), want)
    zero = orc.gated_residual_transposed(r, h, vec(B, D, 0.0))
    assert np.array_equal(zero, r)
    one = orc.gated_residual_transposed(r, h, vec(B, D, 1.0))
    exact = widen(r).astype(np.float64) + np.swapaxes(widen(h), 1, 2).astype(np.float64)
    assert np.array_equal(widen(one), bf16_of_f64(exact).astype(np.float32))


@pytest.mark.parametrize("hd,tree_s", [(128, 16777230.0), (64, 16777222.0)])
def test_qk_head_fold_is_adjacent_pair_tree(orc, hd, tree_s):
    """The head sum folds the hd/8 logical threads' partials by the
    adjacent-pair tree (guide, canonical RMS order; one 8-column chain per
    thread).  Worked by hand: column 0 = 4096 gives thread 0 the partial
    2^24, and column 8l = 1 gives thread l >= 1 the partial 1.  The tree
    adds (2^24 + 1) -> 2^24 (tie to even), then 2^24 + 2, + 4, + 8 for 16
    threads (16777230) or + 2, + 4 for 8 (16777222); a left-to-right sum
    would lose every 1 and give 2^24."""
    H, Tt, Ti = 2, 1, 1
    row = np.zeros(3 * H * hd, np.float32)
    for h in range(2 * H):  # every Q and K head
        base = h * hd
        row[base] = 4096.0
        row[base + 8:base + hd:8] = 1.0
    packed = bits_of(np.stack([row, row]))
    ones = [bits_of(np.ones(hd))] * 4
    eps = 0.0
    _, _, _, rs = orc.qk_norm_rope_epilogue(
        synth.split_qkv(packed[:Tt], H, hd), synth.split_qkv(packed[Tt:], H, hd), H, ones,
        _rope_const_hd(Tt, hd, 1, 0), _rope_const_hd(Ti, hd, 1, 0), eps, eps, with_stats=True,
        head_dim=hd)
    f = np.float32
    want = f(1.0) / np.sqrt(f(tree_s) / f(hd))            # s/hd exact (power of two), eps = 0
    seq = f(1.0) / np.sqrt(f(2.0 ** 24) / f(hd))
    assert want != seq
    assert np.all(rs == want), (rs, want)
