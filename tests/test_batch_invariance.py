"""Batch invariance on the GPU: a row's output bits do not depend on the batch
it is computed in, the token count, padding or the launch shape.

LayerNorm+modulate at D=4096 as a classifier-free-guidance batch (B=2,
T=1140, per-batch scale/shift ~ N(0, 0.2)) is recomputed at B=1 per batch,
row by row (T=1, one launch per row), as one launch of 2280 single-row
batches (vectors read from global memory), and with T padded to 1152
(random pad rows, ignored); every variant must match the full run and the
oracle bit for bit.  The same holds for RMSNorm, the gated form and the QK
epilogue (token subsets of the joint run)."""
import numpy as np
import pytest
import torch

import oracle
from dit_adaln_norm_gb300 import ops, synth
from _gpu import assert_bits_equal, from_dev, to_dev

pytestmark = pytest.mark.gpu
EPS = 1e-6
B, T, TP, D = 2, 1140, 1152, 4096


@pytest.fixture(scope="module")
def cfg_inputs():
    x = synth.outlier_rows_bf16((B, T, D), synth.SEED_X, synth.SEED_OUTLIER)
    vec = synth.normal_bf16((B, 6 * D), synth.SEED_VEC, 0.2)
    sc, sh = vec[:, :D], vec[:, D:2 * D]
    return x, sc, sh


def _variants(fn, x, sc, sh):
    """Outputs [B, T, D] of fn(x, scale, shift) for each batch composition."""
    dsc, dsh = to_dev(np.ascontiguousarray(sc)), to_dev(np.ascontiguousarray(sh))
    out = {"full": from_dev(fn(to_dev(x), dsc, dsh))}
    out["per_batch"] = np.stack([from_dev(fn(to_dev(x[b:b + 1]), dsc[b:b + 1], dsh[b:b + 1]))[0]
                                 for b in range(B)])
    rows = np.empty_like(x)
    for b in range(B):
        xb = to_dev(x[b:b + 1])
        for t in range(T):
            rows[b, t] = from_dev(fn(xb[:, t:t + 1].contiguous(), dsc[b:b + 1], dsh[b:b + 1]))[0, 0]
    out["row_by_row"] = rows
    # one launch, every row its own batch (B*T batches of T=1)
    idx = np.repeat(np.arange(B), T)
    many = fn(to_dev(x.reshape(B * T, 1, D)), dsc[idx], dsh[idx])
    out["single_row_batches"] = from_dev(many).reshape(B, T, D)
    # padded token count
    xp = synth.normal_bf16((B, TP, D), 77, 3.0)
    xp[:, :T] = x
    out["padded"] = from_dev(fn(to_dev(xp), dsc, dsh))[:, :T]
    return out


def test_ln_cfg_batch_invariance(cfg_inputs):
    x, sc, sh = cfg_inputs
    want = oracle.ln_modulate(x, sc, sh, EPS)
    outs = _variants(lambda a, s, h: ops.ln_modulate(a, s, h, EPS), x, sc, sh)
    for name, y in outs.items():
        assert_bits_equal(y, want, f"ln {name}")


def test_rms_batch_invariance(cfg_inputs):
    x, sc, sh = cfg_inputs
    want = oracle.rms_modulate(x, sc, sh, EPS)
    outs = _variants(lambda a, s, h: ops.rms_modulate(a, s, h, EPS), x, sc, sh)
    for name, y in outs.items():
        assert_bits_equal(y, want, f"rms {name}")


def test_gated_batch_invariance(cfg_inputs):
    x, sc, sh = cfg_inputs
    sc, sh = np.ascontiguousarray(sc), np.ascontiguousarray(sh)  # one batch stride with gate
    h = synth.normal_bf16((B, T, D), 5)
    gate = synth.normal_bf16((B, D), 6, 0.1)
    want_r, want_y = oracle.gated_rms_modulate(x, h, gate, sc, sh, EPS)
    dg = to_dev(gate)
    full_r, full_y = ops.gated_rms_modulate(to_dev(x), to_dev(h), dg, to_dev(np.ascontiguousarray(sc)),
                                            to_dev(np.ascontiguousarray(sh)), EPS)
    assert_bits_equal(from_dev(full_r), want_r, "gated r' full")
    assert_bits_equal(from_dev(full_y), want_y, "gated y full")
    for b in range(B):  # per batch, and a token subset of one batch
        for t0, t1 in ((0, T), (17, 530)):
            r_b, y_b = ops.gated_rms_modulate(
                to_dev(x[b:b + 1, t0:t1]), to_dev(h[b:b + 1, t0:t1]), dg[b:b + 1],
                to_dev(np.ascontiguousarray(sc[b:b + 1])), to_dev(np.ascontiguousarray(sh[b:b + 1])),
                EPS)
            assert_bits_equal(from_dev(r_b)[0], want_r[b, t0:t1], f"gated r' b={b} [{t0},{t1})")
            assert_bits_equal(from_dev(y_b)[0], want_y[b, t0:t1], f"gated y b={b} [{t0},{t1})")


def test_qk_token_subsets_match_joint_run():
    H, Tt, Ti = 24, 256, 1024
    pt, pi = synth.packed_qkv(Tt, H, 90), synth.packed_qkv(Ti, H, 91)
    ws = synth.head_weights(4, 92)
    rt, ri = synth.rope_table(Tt), synth.rope_table(Ti, pos0=Tt)
    dw = [to_dev(w) for w in ws]
    Pt, Pi = to_dev(pt), to_dev(pi)
    RT, RI = torch.from_numpy(rt).cuda(), torch.from_numpy(ri).cuda()
    full = [from_dev(o) for o in ops.qk_norm_rope_epilogue(
        synth.split_qkv(Pt, H), synth.split_qkv(Pi, H), *dw, RT, RI, EPS, EPS, H)]
    want = oracle.qk_norm_rope_epilogue(synth.split_qkv(pt, H), synth.split_qkv(pi, H), H, ws,
                                        rt, ri, EPS, EPS)
    for g, w in zip(full, want):
        assert_bits_equal(g, w, "qk joint")
    # image tokens alone (empty text stream), and a slice of each stream
    empty = synth.split_qkv(Pt[:0], H)
    img_only = [from_dev(o) for o in ops.qk_norm_rope_epilogue(
        empty, synth.split_qkv(Pi, H), *dw, RT[:0], RI, EPS, EPS, H)]
    for g, f in zip(img_only, full):
        assert_bits_equal(g, f[Tt:], "qk image only")
    a, b, c, d = 31, 200, 100, 900
    part = [from_dev(o) for o in ops.qk_norm_rope_epilogue(
        synth.split_qkv(Pt[a:b], H), synth.split_qkv(Pi[c:d], H), *dw, RT[a:b].contiguous(),
        RI[c:d].contiguous(), EPS, EPS, H)]
    for g, f in zip(part, full):
        assert_bits_equal(g, np.concatenate([f[a:b], f[Tt + c:Tt + d]]), "qk token slices")


def test_ln_fp8_batch_invariance(cfg_inputs):
    x, sc, sh = cfg_inputs
    qscale = 0.05
    want = oracle.ln_modulate_fp8(x, sc, sh, qscale, EPS)
    dsc, dsh = to_dev(np.ascontiguousarray(sc)), to_dev(np.ascontiguousarray(sh))
    full = ops.ln_modulate_fp8(to_dev(x), dsc, dsh, qscale, EPS).cpu().numpy()
    assert np.array_equal(full, want)
    idx = np.repeat(np.arange(B), T)  # one launch of 2280 single-row batches
    many = ops.ln_modulate_fp8(to_dev(x.reshape(B * T, 1, D)), dsc[idx], dsh[idx], qscale, EPS)
    assert np.array_equal(many.cpu().numpy().reshape(B, T, D), want)
    for b in range(B):
        part = ops.ln_modulate_fp8(to_dev(x[b:b + 1, 40:700]), dsc[b:b + 1], dsh[b:b + 1],
                                   qscale, EPS)
        assert np.array_equal(part.cpu().numpy()[0], want[b, 40:700])


def test_gated_ln_batch_invariance(cfg_inputs):
    x, sc, sh = cfg_inputs
    sc, sh = np.ascontiguousarray(sc), np.ascontiguousarray(sh)
    h = synth.normal_bf16((B, T, D), 7)
    gate = synth.normal_bf16((B, D), 8, 0.1)
    want_r, want_y = oracle.gated_ln_modulate(x, h, gate, sc, sh, EPS)
    dg, dsc, dsh = to_dev(gate), to_dev(sc), to_dev(sh)
    r_all, y_all = ops.gated_ln_modulate(to_dev(x), to_dev(h), dg, dsc, dsh, EPS)
    assert_bits_equal(from_dev(r_all), want_r, "gated ln r' full")
    assert_bits_equal(from_dev(y_all), want_y, "gated ln y full")
    idx = np.repeat(np.arange(B), T)
    r_m, y_m = ops.gated_ln_modulate(to_dev(x.reshape(B * T, 1, D)), to_dev(h.reshape(B * T, 1, D)),
                                     dg[idx], dsc[idx], dsh[idx], EPS)
    assert_bits_equal(from_dev(r_m).reshape(B, T, D), want_r, "gated ln r' single rows")
    assert_bits_equal(from_dev(y_m).reshape(B, T, D), want_y, "gated ln y single rows")


@pytest.mark.parametrize("hd,neox", [(128, True), (64, False), (64, True)])
def test_qk_variant_token_subsets(hd, neox):
    H, Tt, Ti = 24 * 128 // hd, 64, 300
    pt, pi = synth.packed_qkv(Tt, H, 93, hd), synth.packed_qkv(Ti, H, 94, hd)
    ws = synth.head_weights(4, 95, hd)
    rt, ri = synth.rope_table(Tt, hd), synth.rope_table(Ti, hd, pos0=Tt)
    dw = [to_dev(w) for w in ws]
    Pt, Pi = to_dev(pt), to_dev(pi)
    RT, RI = torch.from_numpy(rt).cuda(), torch.from_numpy(ri).cuda()
    run = lambda a, b, ra, rb: [from_dev(o) for o in ops.qk_norm_rope_epilogue(
        synth.split_qkv(a, H, hd), synth.split_qkv(b, H, hd), *dw, ra, rb, EPS, EPS, H,
        head_dim=hd, neox=neox)]
    full = run(Pt, Pi, RT, RI)
    want = oracle.qk_norm_rope_epilogue(synth.split_qkv(pt, H, hd), synth.split_qkv(pi, H, hd),
                                        H, ws, rt, ri, EPS, EPS, head_dim=hd, neox=neox)
    for g, w in zip(full, want):
        assert_bits_equal(g, w, f"qk hd={hd} neox={neox} joint")
    part = run(Pt[5:40], Pi[17:250], RT[5:40].contiguous(), RI[17:250].contiguous())
    for g, f in zip(part, full):
        assert_bits_equal(g, np.concatenate([f[5:40], f[Tt + 17:Tt + 250]]), "qk variant slices")


@pytest.mark.parametrize("kind", ["ln", "rms", "gated", "ln_fp8", "gated_ln"])
def test_launch_shape_invariance(kind):
    """Rows 100..163 of a [1, 4216, 4096] launch (twelve warps per CTA, many
    rows per SM) and the same rows as a [1, 64, 4096] launch (eight warps,
    one row or none per warp) give the same bits."""
    Dm, Tm, lo, hi = 4096, 4216, 100, 164
    x = synth.normal_bf16((1, Tm, Dm), 31)
    h = synth.normal_bf16((1, Tm, Dm), 32)
    vec = to_dev(synth.normal_bf16((1, 6 * Dm), 33, 0.2))
    sc, sh, g = vec[:, :Dm], vec[:, Dm:2 * Dm], vec[:, 2 * Dm:3 * Dm]

    def run(xx, hh):
        if kind == "ln":
            return [ops.ln_modulate(xx, sc, sh, EPS)]
        if kind == "rms":
            return [ops.rms_modulate(xx, sc, sh, EPS)]
        if kind == "ln_fp8":
            return [ops.ln_modulate_fp8(xx, sc, sh, 0.05, EPS)]
        if kind == "gated":
            return list(ops.gated_rms_modulate(xx, hh, g, sc, sh, EPS))
        return list(ops.gated_ln_modulate(xx, hh, g, sc, sh, EPS))

    big = run(to_dev(x), to_dev(h))
    small = run(to_dev(np.ascontiguousarray(x[:, lo:hi])), to_dev(np.ascontiguousarray(h[:, lo:hi])))
    for i, (a, b) in enumerate(zip(big, small)):
        a = a.cpu().view(torch.int16).numpy() if a.dtype == torch.bfloat16 else a.cpu().numpy()
        b = b.cpu().view(torch.int16).numpy() if b.dtype == torch.bfloat16 else b.cpu().numpy()
        assert np.array_equal(a[:, lo:hi], b), f"{kind} output {i}: launch shape changed the bits"
