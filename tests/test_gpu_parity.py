"""GPU parity: the CUDA path through the C ABI against the CPU oracle, bit
for bit (NaN payloads aside), on the same seeded inputs.

Small cases span several CTA row slots with ragged tails; the full-size
cases are the workload shapes of the diffusion sites (FLUX.1 D=3072 image /
text / concat / odd token counts, ERNIE-Image [1,4216,4096], the gated
residual block, the Qwen-Image packed QKV epilogue).  Every output sits
inside sentinel guard bands that must come back untouched."""
import numpy as np
import pytest
import torch

import oracle
from dit_adaln_norm_gb300 import ops, synth
from _gpu import adaln, assert_bits_equal, check_guard, from_dev, guarded, to_dev

pytestmark = pytest.mark.gpu
EPS = 1e-6


@pytest.fixture(scope="module", autouse=True)
def _setup():
    assert torch.cuda.is_available(), "GPU tests need CUDA"
    oracle.build()
    ops.load()


# ------------------------------------------------------------------- RMS

def run_rms(B, T, D, seed, weight=False, chunks=6, x_bits=None, eps=EPS):
    x = synth.normal_bf16((B, T, D), seed) if x_bits is None else x_bits
    (sc, sh), (dsc, dsh) = adaln(B, D, 2, seed + 1, 0.1, chunks)
    w = synth.normal_bf16((D,), seed + 2, 0.1, 1.0) if weight else None
    buf, y = guarded((B, T, D))
    ops.rms_modulate(to_dev(x), dsc, dsh, eps, weight=None if w is None else to_dev(w), out=y)
    torch.cuda.synchronize()
    check_guard(buf)
    want = oracle.rms_modulate(x, sc, sh, eps, weight=w)
    assert_bits_equal(from_dev(y), want, f"rms B={B} T={T} D={D} w={weight}")


@pytest.mark.parametrize("D", [2048, 4096, 6144, 8192])
@pytest.mark.parametrize("weight", [False, True])
def test_rms_small(D, weight):
    run_rms(2, 37, D, 100 + D, weight=weight)


def test_rms_contiguous_vectors_single_batch():
    run_rms(1, 301, 4096, 7, chunks=2)


def test_rms_many_batches_unstaged_vectors():
    # 8 batches x 2 vectors x 4096 x 2 B exceeds the staging budget: the
    # kernel reads bf16(1+scale) and shift from global memory instead.
    run_rms(8, 5, 4096, 8)


def test_rms_config_small_workload():
    """RMSNorm+modulate [1,128,2048], x ~ N(0,1), scale/shift ~ N(0,0.1)."""
    run_rms(1, 128, 2048, synth.SEED_X)


def test_rms_metric_shape():
    run_rms(1, 4216, 4096, synth.SEED_X)


def test_rms_wide_rows_shared_by_warps():
    # rows of 8192 are split over a team of warps: several rows per team
    run_rms(1, 2000, 8192, 11, weight=True)


# ------------------------------------------------------------- gated RMS

def run_gated(B, T, D, seed, weight=False, inplace=False, chunks=6):
    r = synth.normal_bf16((B, T, D), seed)
    h = synth.normal_bf16((B, T, D), seed + 1)
    (g, sc, sh), (dg, dsc, dsh) = adaln(B, D, 3, seed + 2, 0.1, chunks)
    w = synth.normal_bf16((D,), seed + 3, 0.1, 1.0) if weight else None
    dr = to_dev(r)
    buf, y = guarded((B, T, D))
    if inplace:
        r_out = dr
    else:
        rbuf, r_out = guarded((B, T, D))
    ops.gated_rms_modulate(dr, to_dev(h), dg, dsc, dsh, EPS,
                           weight=None if w is None else to_dev(w), r_out=r_out, out=y)
    torch.cuda.synchronize()
    check_guard(buf)
    if not inplace:
        check_guard(rbuf)
    want_r, want_y = oracle.gated_rms_modulate(r, h, g, sc, sh, EPS, weight=w)
    assert_bits_equal(from_dev(r_out), want_r, f"gated r' D={D}")
    assert_bits_equal(from_dev(y), want_y, f"gated y D={D}")


@pytest.mark.parametrize("D", [2048, 4096, 6144, 8192])
@pytest.mark.parametrize("weight", [False, True])
def test_gated_small(D, weight):
    run_gated(2, 29, D, 200 + D, weight=weight)


def test_gated_in_place_residual():
    run_gated(1, 53, 4096, 300, inplace=True)


def test_gated_many_batches_unstaged_vectors():
    run_gated(5, 6, 4096, 301)


def test_gated_wide_rows_shared_by_warps():
    run_gated(1, 1500, 8192, 12)


def test_gated_config():
    """Gated residual [1,4216,4096]: r, h ~ N(0,1); gate/scale/shift ~ N(0,0.1)."""
    run_gated(1, 4216, 4096, synth.SEED_X)


# ------------------------------------------------------------- LayerNorm

def run_ln(B, T, D, seed, outliers=False, chunks=6, x_bits=None, eps=EPS, in_place=False,
           std=0.2):
    if x_bits is not None:
        x = x_bits
    elif outliers:
        x = synth.outlier_rows_bf16((B, T, D), seed, synth.SEED_OUTLIER)
    else:
        x = synth.normal_bf16((B, T, D), seed)
    (sc, sh), (dsc, dsh) = adaln(B, D, 2, seed + 1, std, chunks)
    if in_place:
        y = to_dev(x)
        ops.ln_modulate(y, dsc, dsh, eps, out=y)
    else:
        buf, y = guarded((B, T, D))
        ops.ln_modulate(to_dev(x), dsc, dsh, eps, out=y)
    torch.cuda.synchronize()
    if not in_place:
        check_guard(buf)
    want = oracle.ln_modulate(x, sc, sh, eps)
    assert_bits_equal(from_dev(y), want, f"ln B={B} T={T} D={D}")


@pytest.mark.parametrize("D", [8, 64, 1040, 2048, 3072, 4096, 5000, 6144, 8192])
def test_ln_small(D):
    run_ln(2, 41, D, 400 + D, outliers=D >= 1024)


def test_ln_in_place():
    run_ln(1, 77, 3072, 401, outliers=True, in_place=True)


def test_ln_many_batches_unstaged_vectors():
    run_ln(9, 4, 3072, 402)


@pytest.mark.parametrize("T", [4096, 512, 4608, 4093])
def test_ln_flux_site_configs(T):
    """FLUX.1-like sites, D=3072: x ~ N(0,1) with 1% of channels x20,
    scale/shift ~ N(0,0.2); image, text, concat and odd token counts."""
    run_ln(1, T, 3072, synth.SEED_X, outliers=True)


def test_ln_metric_shape():
    run_ln(1, 4216, 4096, synth.SEED_X, outliers=True)


def test_ln_flux_cfg_site_odd_tokens():
    """The FLUX LayerNorm test's CFG case: [2, 300, 3072], x = N(0,1) * 8,
    scale/shift chunk views of a 6-chunk embedding."""
    run_ln(2, 300, 3072, 403, x_bits=synth.normal_bf16((2, 300, 3072), 403, 8.0), chunks=6)


# ------------------------------------------------------------ edge cases

def _special_rows(D, seed):
    rng = np.random.Generator(np.random.PCG64(seed))
    rows = [np.zeros(D), np.full(D, 3.0), np.full(D, -1e-30),
            rng.standard_normal(D) * 1e30, rng.standard_normal(D) * 1e-38,
            rng.standard_normal(D) * 1e-42,                       # bf16 subnormals
            np.where(np.arange(D) % 2, 1.0, -1.0), rng.standard_normal(D) * 3e38]
    r = rng.standard_normal(D)
    r[5] = np.inf
    rows.append(r)
    r = rng.standard_normal(D)
    r[D // 2] = -np.inf
    rows.append(r)
    r = rng.standard_normal(D)
    r[7] = np.nan
    rows.append(r)
    r = rng.standard_normal(D)
    r[: D // 2] *= 1e20
    rows.append(r)
    return synth.to_bf16_bits(np.stack(rows).astype(np.float32))[None]


@pytest.mark.parametrize("eps", [EPS, 0.0])
def test_extreme_rows_rms(eps):
    D = 4096
    run_rms(1, 12, D, 500, x_bits=_special_rows(D, 501), eps=eps)


@pytest.mark.parametrize("eps", [EPS, 0.0])
def test_extreme_rows_ln(eps):
    for D in (3072, 4096):
        run_ln(1, 12, D, 502, x_bits=_special_rows(D, 503), eps=eps)


def test_extreme_vectors():
    """scale = -1 (o = 0), huge and tiny scale/shift values."""
    B, T, D = 1, 16, 2048
    x = synth.normal_bf16((B, T, D), 510)
    rng = np.random.Generator(np.random.PCG64(511))
    sc = synth.to_bf16_bits(np.where(rng.random(D) < 0.3, -1.0,
                                     rng.standard_normal(D) * 1e4).astype(np.float32))[None]
    sh = synth.to_bf16_bits((rng.standard_normal(D) * 1e-30).astype(np.float32))[None]
    y = ops.rms_modulate(to_dev(x), to_dev(sc), to_dev(sh), EPS)
    assert_bits_equal(from_dev(y), oracle.rms_modulate(x, sc, sh, EPS), "rms extreme vectors")
    y = ops.ln_modulate(to_dev(x), to_dev(sc), to_dev(sh), EPS)
    assert_bits_equal(from_dev(y), oracle.ln_modulate(x, sc, sh, EPS), "ln extreme vectors")


def test_empty_inputs_touch_nothing():
    D = 4096
    x = torch.empty((1, 0, D), dtype=torch.bfloat16, device="cuda")
    v = torch.zeros((1, D), dtype=torch.bfloat16, device="cuda")
    assert ops.rms_modulate(x, v, v, EPS).shape == (1, 0, D)
    assert ops.ln_modulate(x, v, v, EPS).shape == (1, 0, D)
    r_out, y = ops.gated_rms_modulate(x, x, v, v, v, EPS)
    assert y.shape == (1, 0, D)


def test_invalid_arguments_raise_before_launch():
    D = 4096
    x = torch.zeros((1, 8, D), dtype=torch.bfloat16, device="cuda")
    v = torch.zeros((1, D), dtype=torch.bfloat16, device="cuda")
    with pytest.raises(ops.DanError) as e:
        ops.rms_modulate(x[:, :, :3072].contiguous(), v[:, :3072], v[:, :3072], EPS)
    assert e.value.status == ops.DAN_EUNSUPPORTED
    with pytest.raises(ops.DanError) as e:
        ops.rms_modulate(x, v, v, -1.0)
    assert e.value.status == ops.DAN_EINVAL
    big = torch.zeros((2, 8, D), dtype=torch.bfloat16, device="cuda")
    with pytest.raises(ops.DanError) as e:  # output overlapping half of the input
        ops.ln_modulate(big[:1], v, v, EPS, out=big.view(-1)[8 * D // 2:][:8 * D].view(1, 8, D))
    assert e.value.status == ops.DAN_EALIAS


# ------------------------------------------------------- QK epilogue

def run_qk(Tt, Ti, H, seed, packed=True, eps=(1e-6, 1e-6), hd=128, neox=False):
    pt = synth.packed_qkv(Tt, H, seed, hd)
    pi = synth.packed_qkv(Ti, H, seed + 1, hd)
    ws = synth.head_weights(4, seed + 2, hd)
    rt, ri = synth.rope_table(Tt, hd), synth.rope_table(Ti, hd, pos0=Tt)
    if packed:
        Pt, Pi = to_dev(pt), to_dev(pi)
        dt, di = synth.split_qkv(Pt, H, hd), synth.split_qkv(Pi, H, hd)
    else:
        dt = tuple(to_dev(a) for a in synth.split_qkv(pt, H, hd))
        di = tuple(to_dev(a) for a in synth.split_qkv(pi, H, hd))
    dw = [to_dev(w) for w in ws]
    bufs, outs = zip(*[guarded((Tt + Ti, H, hd)) for _ in range(3)])
    ops.qk_norm_rope_epilogue(dt, di, *dw, torch.from_numpy(rt).cuda(),
                              torch.from_numpy(ri).cuda(), eps[0], eps[1], H, out=outs,
                              head_dim=hd, neox=neox)
    torch.cuda.synchronize()
    for b in bufs:
        check_guard(b)
    want = oracle.qk_norm_rope_epilogue(synth.split_qkv(pt, H, hd), synth.split_qkv(pi, H, hd),
                                        H, ws, rt, ri, eps[0], eps[1], head_dim=hd, neox=neox)
    for name, g, w in zip("qkv", outs, want):
        assert_bits_equal(from_dev(g), w, f"qk {name} Tt={Tt} Ti={Ti} H={H} hd={hd} neox={neox}")


@pytest.mark.parametrize("hd", [128, 64])
def test_qk_head_fold_order_case(hd):
    """Heads whose sum depends on the fold order (thread 0's partial 2^24,
    the others 1: the adjacent-pair tree keeps the 1s a left-to-right sum
    loses), among random heads."""
    H, Tt, Ti = 24 * 128 // hd, 3, 5
    pt, pi = synth.packed_qkv(Tt, H, 640, hd), synth.packed_qkv(Ti, H, 641, hd)
    special = np.zeros(hd, np.float32)
    special[0] = 4096.0
    special[8::8] = 1.0
    for arr in (pt, pi):
        for h in range(0, 2 * H, 3):  # every third Q/K head
            arr[:, h * hd:(h + 1) * hd] = synth.to_bf16_bits(special)
    ws = [synth.to_bf16_bits(np.ones(hd, np.float32))] * 4
    rt, ri = synth.rope_table(Tt, hd), synth.rope_table(Ti, hd, pos0=Tt)
    Pt, Pi = to_dev(pt), to_dev(pi)
    outs = ops.qk_norm_rope_epilogue(synth.split_qkv(Pt, H, hd), synth.split_qkv(Pi, H, hd),
                                     *[to_dev(w) for w in ws], torch.from_numpy(rt).cuda(),
                                     torch.from_numpy(ri).cuda(), 0.0, 0.0, H, head_dim=hd)
    want = oracle.qk_norm_rope_epilogue(synth.split_qkv(pt, H, hd), synth.split_qkv(pi, H, hd),
                                        H, ws, rt, ri, 0.0, 0.0, head_dim=hd)
    for name, g, w in zip("qkv", outs, want):
        assert_bits_equal(from_dev(g), w, f"qk fold-order case {name} hd={hd}")


# ------------------------------ hand-worked operand-order probes on the GPU

def _golden(name, probe):
    import json
    import os
    path = os.path.join(os.path.dirname(__file__), "golden", name)
    return {p["name"]: p for p in json.load(open(path))["probes"]}[probe]


def _widen(bits):
    return (np.asarray(bits).astype(np.uint32) << 16).view(np.float32)


def test_rms_weight_product_order_probe():
    """The probe row (tests/golden, rms_weight_product_order: the weight
    multiplies rn(x*rstd), which puts one column on a bf16 tie) among random
    rows; GPU == hand-worked values == oracle."""
    p = _golden("rounding_boundary_probes.json", "rms_weight_product_order")
    D, T = p["D"], 40
    x = synth.normal_bf16((1, T, D), 650)
    probe = synth.to_bf16_bits(np.tile(np.asarray(p["x_alternating"], np.float32), D // 2))
    x[0, ::7] = probe
    zero = np.zeros((1, D), np.uint16)
    w = synth.to_bf16_bits(np.full(D, p["weight"], np.float32))
    buf, y = guarded((1, T, D))
    ops.rms_modulate(to_dev(x), to_dev(zero), to_dev(zero), p["eps"], weight=to_dev(w), out=y)
    torch.cuda.synchronize()
    check_guard(buf)
    got = from_dev(y)
    expect = np.tile(np.asarray(p["expected_y_alternating"], np.float32), D // 2)
    assert np.array_equal(_widen(got[0, ::7]), np.broadcast_to(expect, got[0, ::7].shape))
    assert_bits_equal(got, oracle.rms_modulate(x, zero, zero, p["eps"], weight=w), "rms probe")


def test_qk_weight_product_order_probe():
    """Heads of the qk_weight_product_order probe (rn(rn(x*rstd)*w) puts one
    column on a bf16 tie) at every third Q/K head among random heads, with
    the identity rotation; GPU == hand-worked values == oracle."""
    p = _golden("rounding_boundary_probes.json", "qk_weight_product_order")
    hd, H, Tt, Ti = p["head_dim"], 24, 3, 5
    pt, pi = synth.packed_qkv(Tt, H, 660, hd), synth.packed_qkv(Ti, H, 661, hd)
    head = synth.to_bf16_bits(np.tile(np.asarray(p["x_alternating"], np.float32), hd // 2))
    for arr in (pt, pi):
        for h in range(0, 2 * H, 3):
            arr[:, h * hd:(h + 1) * hd] = head
    ws = [synth.to_bf16_bits(np.full(hd, p["weight"], np.float32))] * 4
    rope = lambda T: np.concatenate([np.full((T, hd // 2), p["cos"], np.float32),
                                     np.full((T, hd // 2), p["sin"], np.float32)], 1)
    Pt, Pi = to_dev(pt), to_dev(pi)
    outs = ops.qk_norm_rope_epilogue(synth.split_qkv(Pt, H, hd), synth.split_qkv(Pi, H, hd),
                                     *[to_dev(w) for w in ws], torch.from_numpy(rope(Tt)).cuda(),
                                     torch.from_numpy(rope(Ti)).cuda(), p["eps"], p["eps"], H,
                                     head_dim=hd)
    got = [from_dev(g) for g in outs]
    expect = np.tile(np.asarray(p["expected_alternating"], np.float32), hd // 2)
    for h in range(0, 2 * H, 3):
        src = got[0] if h < H else got[1]
        assert np.array_equal(_widen(src[:, h % H]), np.broadcast_to(expect, (Tt + Ti, hd)))
    want = oracle.qk_norm_rope_epilogue(synth.split_qkv(pt, H, hd), synth.split_qkv(pi, H, hd),
                                        H, ws, rope(Tt), rope(Ti), p["eps"], p["eps"],
                                        head_dim=hd)
    for name, g, w in zip("qkv", got, want):
        assert_bits_equal(g, w, f"qk weight-order probe {name}")


def test_ln_combine_count_weighting_probe():
    """The combine_count_weighting probe row (D = 40: states of 24 and 16
    elements merge; the count weighting decides one bf16 step of the x = 2
    outputs at this eps) among random rows; GPU == hand-worked == oracle."""
    p = _golden("ln_order_probes.json", "combine_count_weighting")
    D, T = p["D"], 50
    x = synth.normal_bf16((1, T, D), 670)
    runs = lambda rr: np.concatenate([np.full(n, v, np.float32) for v, n in rr])
    x[0, ::5] = synth.to_bf16_bits(runs(p["x_runs"]))
    zero = np.zeros((1, D), np.uint16)
    buf, y = guarded((1, T, D))
    ops.ln_modulate(to_dev(x), to_dev(zero), to_dev(zero), p["eps"], out=y)
    torch.cuda.synchronize()
    check_guard(buf)
    got = from_dev(y)
    expect = runs([(v, n) for v, (_, n) in zip(p["expected_y_runs"], p["x_runs"])])
    assert np.array_equal(_widen(got[0, ::5]), np.broadcast_to(expect, got[0, ::5].shape))
    assert_bits_equal(got, oracle.ln_modulate(x, zero, zero, p["eps"]), "ln combine probe")


def _probes(name):
    import json
    import os
    path = os.path.join(os.path.dirname(__file__), "golden", name)
    return json.load(open(path))["probes"]


@pytest.mark.parametrize("probe", [p["name"] for p in _probes("ln_order_probes.json")])
def test_ln_order_probe_rows(probe):
    """Every hand-worked LayerNorm order probe row among random rows at its
    own width and eps: GPU == oracle bit for bit."""
    p = _golden("ln_order_probes.json", probe)
    D, T = p["D"], 20
    runs = lambda rr: np.concatenate([np.full(n, v, np.float32) for v, n in rr])
    row = np.asarray(p["x"], np.float32) if "x" in p else runs(p["x_runs"])
    x = synth.normal_bf16((1, T, D), 680)
    x[0, 1::6] = synth.to_bf16_bits(row)
    zero = np.zeros((1, D), np.uint16)
    y = torch.empty((1, T, D), dtype=torch.bfloat16, device="cuda")
    ops.ln_modulate(to_dev(x), to_dev(zero), to_dev(zero), p["eps"], out=y)
    torch.cuda.synchronize()
    assert_bits_equal(from_dev(y), oracle.ln_modulate(x, zero, zero, p["eps"]), probe)


@pytest.mark.parametrize("probe", [p["name"] for p in _probes("rms_order_probes.json")])
def test_rms_order_probe_rows(probe):
    """Every hand-worked RMS order probe row among random rows: GPU == oracle."""
    p = _golden("rms_order_probes.json", probe)
    D, T = p["D"], 20
    row = np.zeros(D, np.float32)
    cols = p["columns"]
    if "ones_thread" in cols:
        tpr = D // 64
        for b in range(8):
            row[8 * tpr * b + 8 * cols["ones_thread"]:][:8] = 1.0
    for c, val in cols["big"]:
        row[c] = val
    x = synth.normal_bf16((1, T, D), 681)
    x[0, 2::5] = synth.to_bf16_bits(row)
    zero = np.zeros((1, D), np.uint16)
    eps = p.get("eps", EPS)
    y = torch.empty((1, T, D), dtype=torch.bfloat16, device="cuda")
    ops.rms_modulate(to_dev(x), to_dev(zero), to_dev(zero), eps, out=y)
    torch.cuda.synchronize()
    assert_bits_equal(from_dev(y), oracle.rms_modulate(x, zero, zero, eps), probe)


@pytest.mark.parametrize("H", [24, 3, 1, 30])
@pytest.mark.parametrize("packed", [True, False])
def test_qk_small(H, packed):
    run_qk(7, 33, H, 600 + H, packed=packed, eps=(1e-6, 1e-5))


def test_qk_one_stream_empty():
    run_qk(0, 19, 24, 610)
    run_qk(11, 0, 24, 611)


def test_qk_config():
    """Qwen-Image packed QKV: 256 text + 4096 image tokens, 24 heads x 128."""
    run_qk(256, 4096, 24, synth.SEED_X)


@pytest.mark.parametrize("hd,neox", [(64, False), (64, True), (128, True)])
@pytest.mark.parametrize("H", [1, 5, 24, 48, 50])
def test_qk_variants_small(hd, neox, H):
    run_qk(5, 29, H, 620 + H + hd, packed=H % 2 == 0, eps=(1e-6, 1e-5), hd=hd, neox=neox)


@pytest.mark.parametrize("hd,neox", [(64, False), (64, True), (128, True)])
def test_qk_variants_config(hd, neox):
    run_qk(256, 4096, 24 if hd == 128 else 48, synth.SEED_X + 7, hd=hd, neox=neox)


def test_signed_zeros_through_the_modulate_chain():
    """-0 inputs give n = -0; with scale = 0 the product keeps its sign and
    -0 + -0 = -0 must come out, while -0 + +0 = +0."""
    B, T, D = 1, 6, 4096
    rng = np.random.Generator(np.random.PCG64(520))
    x = synth.normal_bf16((B, T, D), 521)
    x[0, :3, ::3] = 0x8000          # -0 entries in normal rows
    x[0, 3] = 0x8000                # a row of -0 (eps > 0: rstd finite)
    x[0, 4] = 0x0000                # a row of +0
    sh = synth.normal_bf16((B, D), 522, 0.1)
    sh[0, rng.random(D) < 0.5] = 0x8000
    sh[0, ::7] = 0x0000
    sc = np.zeros((B, D), np.uint16)
    sc[0, 1::5] = 0x8000            # scale = -0 -> o = 1
    for fn in (oracle.rms_modulate, oracle.ln_modulate):
        want = fn(x, sc, sh, EPS)
        got = (ops.rms_modulate if fn is oracle.rms_modulate else ops.ln_modulate)(
            to_dev(x), to_dev(sc), to_dev(sh), EPS)
        assert_bits_equal(from_dev(got), want, "signed zeros")
    g = np.zeros((B, D), np.uint16)
    g[0, ::2] = 0x8000              # gate = -0: gate*h = -+0, r + that
    r = x.copy()
    wr, wy = oracle.gated_rms_modulate(r, x, g, sc, sh, EPS)
    gr, gy = ops.gated_rms_modulate(to_dev(r), to_dev(x), to_dev(g), to_dev(sc), to_dev(sh), EPS)
    assert_bits_equal(from_dev(gr), wr, "signed zeros gated r'")
    assert_bits_equal(from_dev(gy), wy, "signed zeros gated y")


# ------------------------------------------------ LayerNorm + modulate + FP8

def run_ln_fp8(B, T, D, seed, qscale, outliers=True, chunks=6, x_bits=None):
    if x_bits is not None:
        x = x_bits
    elif outliers:
        x = synth.outlier_rows_bf16((B, T, D), seed, synth.SEED_OUTLIER)
    else:
        x = synth.normal_bf16((B, T, D), seed)
    (sc, sh), (dsc, dsh) = adaln(B, D, 2, seed + 1, 0.2, chunks)
    total = B * T * D
    buf = torch.full((total + 2 * 4096,), 0xA5, dtype=torch.uint8, device="cuda")
    q = buf[4096:4096 + total].view(B, T, D)
    ops.ln_modulate_fp8(to_dev(x), dsc, dsh, qscale, EPS, out=q)
    torch.cuda.synchronize()
    assert bool((buf[:4096] == 0xA5).all()) and bool((buf[4096 + total:] == 0xA5).all())
    want = oracle.ln_modulate_fp8(x, sc, sh, qscale, EPS)
    got = q.cpu().numpy()
    nan = lambda c: (c & 0x7F) == 0x7F
    same = (got == want) | (nan(got) & nan(want))
    assert same.all(), (f"ln_fp8 B={B} T={T} D={D} qscale={qscale}: {int((~same).sum())} codes "
                        f"differ, first at {np.argwhere(~same)[0]}")


@pytest.mark.parametrize("D", [8, 1040, 2048, 3072, 4096, 5000, 8192])
def test_ln_fp8_small(D):
    run_ln_fp8(2, 19, D, 400 + D, 0.05)


@pytest.mark.parametrize("qscale", [1.0, 0.0078125, 0.003, 7.5])
def test_ln_fp8_scales_and_saturation(qscale):
    # small scales push most codes into saturation at +-448
    run_ln_fp8(1, 257, 3072, 410, qscale)


def test_ln_fp8_extreme_rows():
    D = 1024
    rows = [np.zeros(D), np.full(D, 3.0), np.where(np.arange(D) % 2 == 0, 1e4, -1e4),
            np.linspace(-1e-30, 1e-30, D), np.random.default_rng(411).normal(0, 50, D)]
    x = np.stack([synth.to_bf16_bits(np.asarray(r, np.float32)) for r in rows])[None]
    run_ln_fp8(1, len(rows), D, 412, 0.1, x_bits=x)


def test_ln_fp8_metric_shape_and_cfg_batch():
    run_ln_fp8(1, 4216, 4096, synth.SEED_X, 0.05)
    run_ln_fp8(2, 1140, 4096, synth.SEED_X + 1, 0.05)


# ------------------------------------- rows of several batches per team

@pytest.mark.parametrize("B,T", [(3, 1300), (5, 777)])
def test_rows_across_batches(B, T):
    """Enough rows for the twelve-warp shapes, with fewer tokens per batch
    than the rows between two of a team's rows in the interleaved order (152
    CTAs x 12 teams), so a team's batch index advances by one or two batches
    per row."""
    run_rms(B, T, 4096, 620 + T)
    run_rms(B, T, 8192, 621 + T, weight=True)
    run_gated(B, T, 4096, 622 + T)
    run_ln(B, T, 4096, 623 + T, outliers=True)
    run_ln(B, T, 3072, 624 + T)
    run_ln_fp8(B, T, 4096, 625 + T, 0.05)
    run_gated_ln(B, T, 3072, 626 + T)


# ------------------------------------------------ gated residual + LayerNorm

def run_gated_ln(B, T, D, seed, inplace=False, chunks=6):
    r = synth.outlier_rows_bf16((B, T, D), seed, synth.SEED_OUTLIER)
    h = synth.normal_bf16((B, T, D), seed + 1)
    (g, sc, sh), (dg, dsc, dsh) = adaln(B, D, 3, seed + 2, 0.1, chunks)
    dr = to_dev(r)
    buf, y = guarded((B, T, D))
    if inplace:
        r_out = dr
    else:
        rbuf, r_out = guarded((B, T, D))
    ops.gated_ln_modulate(dr, to_dev(h), dg, dsc, dsh, EPS, r_out=r_out, out=y)
    torch.cuda.synchronize()
    check_guard(buf)
    if not inplace:
        check_guard(rbuf)
    want_r, want_y = oracle.gated_ln_modulate(r, h, g, sc, sh, EPS)
    assert_bits_equal(from_dev(r_out), want_r, f"gated ln r' D={D}")
    assert_bits_equal(from_dev(y), want_y, f"gated ln y D={D}")


@pytest.mark.parametrize("D", [8, 1040, 3072, 4096, 5000, 8192])
def test_gated_ln_small(D):
    run_gated_ln(2, 23, D, 500 + D)


def test_gated_ln_in_place_and_shapes():
    run_gated_ln(1, 97, 3072, 510, inplace=True)
    run_gated_ln(1, 4216, 4096, synth.SEED_X)
    run_gated_ln(2, 1140, 4096, synth.SEED_X + 2)


# ---------------------------------- residual gating in the transposed layout

def run_resid_t(B, D, T, seed, inplace=False):
    r = synth.normal_bf16((B, D, T), seed)
    h = synth.normal_bf16((B, T, D), seed + 1)
    emb = synth.normal_bf16((B, 6 * D), seed + 2, 0.5)
    g = emb[:, 2 * D:3 * D]
    dg = to_dev(emb)[:, 2 * D:3 * D]
    dr = to_dev(r)
    if inplace:
        out = dr
    else:
        buf, out = guarded((B, D, T))
    ops.gated_residual_transposed(dr, to_dev(h), dg, out=out)
    torch.cuda.synchronize()
    if not inplace:
        check_guard(buf)
    assert_bits_equal(from_dev(out), oracle.gated_residual_transposed(r, h, g),
                      f"resid_t B={B} D={D} T={T}")


@pytest.mark.parametrize("B,D,T", [(1, 8, 1), (1, 72, 37), (2, 64, 64), (1, 136, 130),
                                   (2, 3072, 97), (1, 256, 4093), (1, 8, 8), (1, 72, 136),
                                   (2, 200, 8), (3, 520, 72), (1, 8, 3), (1, 16, 2),
                                   (3, 24, 65), (1, 64, 63), (2, 40, 127), (1, 1032, 4094)])
def test_gated_residual_transposed_shapes(B, D, T):
    run_resid_t(B, D, T, 700 + D + T)


def test_gated_residual_transposed_in_place_and_site():
    run_resid_t(1, 3072, 4096, 710, inplace=True)
    run_resid_t(2, 3072, 512, 711)


def test_gated_residual_transposed_tile_runs_cross_batches():
    """More tiles than resident CTAs, with ragged channel and token tiles:
    a CTA's run of tiles crosses a batch boundary and reuses its stages."""
    run_resid_t(2, 1032, 1800, 712)
    run_resid_t(2, 1032, 1800, 713, inplace=True)


def test_gated_residual_transposed_odd_tokens():
    """T odd: the residual rows of odd channels start on odd elements, so the
    tile's token pairs and its single edge tokens change with the channel;
    in place, across batches with ragged tiles, and at the [1,3072,4093]
    workload."""
    run_resid_t(2, 1032, 1799, 714)
    run_resid_t(2, 1032, 1799, 715, inplace=True)
    run_resid_t(1, 136, 129, 716, inplace=True)
    run_resid_t(1, 3072, 4093, 717)
