"""Host-side tests of the C ABI (no GPU): the library loads, exports every
function include/dan.h declares, and each dan_can_use_* returns the
documented status.  The pointers here are fake addresses: validation only
inspects their values, never dereferences them."""
import ctypes
import os

import pytest

from dit_adaln_norm_gb300 import build as dan_build
from dit_adaln_norm_gb300 import ops

OK, EINVAL, EUNSUP, EALIGN, EALIAS, ECUDA = range(6)
MB = 1 << 20
EPS = 1e-6


@pytest.fixture(scope="module")
def lib():
    dan_build.build()
    return ops.load()


def test_exports_every_declared_symbol(lib):
    names = ops.declared_symbols()
    assert len(names) == 20
    for n in names:
        assert hasattr(lib, n), n


def test_status_strings(lib):
    for s in range(6):
        assert ops.status_string(s).startswith("DAN_")
    assert "unknown" in ops.status_string(42)


# fake, well-separated device addresses (16-byte aligned)
X, Y, SC, SH, W, R, H, G, RO = (0x10000000 + i * 256 * MB for i in range(9))


def rms(x=X, w=None, sc=SC, sh=SH, vs=4096, y=Y, B=1, T=4216, D=4096, eps=EPS, lib=None):
    return lib.dan_can_use_rms_modulate(x, w, sc, sh, vs, y, B, T, D, eps)


def test_rms_validation(lib):
    f = lambda **k: rms(lib=lib, **k)
    assert f() == OK
    assert f(w=W) == OK
    for D in (2048, 6144, 8192):
        assert f(D=D, vs=D) == OK
    for D in (0, 1024, 3072, 4097, 10240, 16384):
        assert f(D=D, vs=max(D, 8)) == EUNSUP
    assert f(B=-1) == EINVAL and f(T=-3) == EINVAL
    assert f(eps=-1e-6) == EINVAL and f(eps=float("nan")) == EINVAL and f(eps=float("inf")) == EINVAL
    assert f(x=None) == EINVAL and f(y=None) == EINVAL and f(sc=None) == EINVAL
    assert f(x=X + 8) == EALIGN and f(y=Y + 2) == EALIGN and f(w=W + 4) == EALIGN
    assert f(B=2, vs=4100) == EALIGN
    assert f(B=2, vs=4000) == EINVAL  # vs < D
    assert f(B=2, vs=6 * 4096) == OK  # chunk(6) view of an embedding
    # empty problems validate the rest and launch nothing
    assert f(T=0, x=None, y=None) == OK and f(B=0) == OK
    # in place is allowed, partial overlap is not
    assert f(y=X) == OK
    assert f(y=X + 4096) == EALIAS
    assert f(y=SC) == EALIAS and f(w=Y + 64) == EALIAS
    assert f(sh=Y + 4216 * 4096 * 2 - 64) == EALIAS  # vector inside the output
    assert f(sh=Y + 4216 * 4096 * 2) == OK           # right after it


def test_gated_validation(lib):
    def f(r=R, h=H, g=G, w=None, sc=SC, sh=SH, vs=4096, ro=RO, y=Y, B=1, T=4216, D=4096, eps=EPS):
        return lib.dan_can_use_gated_rms_modulate(r, h, g, w, sc, sh, vs, ro, y, B, T, D, eps)

    assert f() == OK and f(w=W) == OK
    assert f(ro=R) == OK               # residual updated in place
    assert f(y=R) == EALIAS            # y may not overwrite an input
    assert f(ro=H) == EALIAS           # r_out may not overwrite h
    assert f(y=RO) == EALIAS           # outputs disjoint
    assert f(ro=R + 64) == EALIAS
    assert f(D=3072, vs=3072) == EUNSUP
    assert f(g=None) == EINVAL and f(h=G + 1) == EALIGN


def test_ln_validation(lib):
    def f(x=X, sc=SC, sh=SH, vs=3072, y=Y, B=1, T=4096, D=3072, eps=EPS):
        return lib.dan_can_use_ln_modulate(x, sc, sh, vs, y, B, T, D, eps)

    for D in (8, 16, 1040, 3072, 4096, 5000, 8192):
        assert f(D=D, vs=D) == OK, D
    for D in (0, 4, 12, 8200, 16384):
        assert f(D=D, vs=max(D, 8)) == EUNSUP, D
    assert f(y=X) == OK and f(y=X + 16) == EALIAS
    assert f(B=2, vs=6 * 3072) == OK and f(B=2, vs=3076) == EALIGN


def test_gated_ln_validation(lib):
    def f(r=R, h=H, g=G, sc=SC, sh=SH, vs=3072, ro=RO, y=Y, B=1, T=4096, D=3072, eps=EPS):
        return lib.dan_can_use_gated_ln_modulate(r, h, g, sc, sh, vs, ro, y, B, T, D, eps)

    assert f() == OK and f(D=1040, vs=1040) == OK
    assert f(ro=R) == OK               # residual updated in place
    assert f(y=R) == EALIAS and f(ro=H) == EALIAS and f(y=RO) == EALIAS
    assert f(D=12, vs=16) == EUNSUP and f(g=None) == EINVAL and f(h=G + 8) == EALIGN


def test_gated_residual_transposed_validation(lib):
    def f(r=R, h=H, g=G, vs=3072, ro=RO, B=1, T=4096, D=3072):
        return lib.dan_can_use_gated_residual_transposed(r, h, g, vs, ro, B, T, D)

    assert f() == OK and f(T=4093) == OK and f(ro=R) == OK
    assert f(D=12, vs=16) == EUNSUP and f(D=0, vs=8) == EUNSUP
    assert f(ro=H) == EALIAS and f(ro=R + 64) == EALIAS
    assert f(h=H + 8) == EALIGN and f(B=2, vs=3076) == EALIGN and f(B=2, vs=3000) == EINVAL
    assert f(g=None) == EINVAL and f(T=0, r=None, h=None, ro=None) == OK


def test_ln_fp8_validation(lib):
    def f(x=X, sc=SC, sh=SH, vs=4096, qs=0.5, q=Y, B=1, T=4216, D=4096, eps=EPS):
        return lib.dan_can_use_ln_modulate_fp8(x, sc, sh, vs, qs, q, B, T, D, eps)

    assert f() == OK and f(D=3072, vs=3072) == OK
    for qs in (0.0, -1.0, float("inf"), float("nan")):
        assert f(qs=qs) == EINVAL
    assert f(q=None) == EINVAL and f(q=Y + 8) == EALIGN
    assert f(q=X) == EALIAS                      # no in-place form
    assert f(q=X + 4216 * 4096 * 2) == OK        # right after x
    assert f(D=12, vs=16) == EUNSUP
    assert f(T=0, x=None, q=None) == OK


def test_qk_validation(lib):
    QT, QI, WT, RT, RI, QO, KO, VO = (0x10000000 + i * 256 * MB for i in range(8))
    Tt, Ti, Hh = 256, 4096, 24
    S = 3 * Hh * 128

    def f(qt=QT, Tt=Tt, st=S, qi=QI, Ti=Ti, si=S, heads=Hh, hd=128, wt=WT, rt=RT, ri=RI,
          eps_t=EPS, eps_i=EPS, qo=QO, ko=KO, vo=VO):
        w = Hh * 128 * 2
        return lib.dan_can_use_qk_norm_rope_epilogue(
            qt, qt + w if qt else None, qt + 2 * w if qt else None, Tt, st,
            qi, qi + w if qi else None, qi + 2 * w if qi else None, Ti, si, heads, hd,
            wt, wt + 256, wt + 512, wt + 768, rt, ri, eps_t, eps_i, qo, ko, vo)

    assert f() == OK
    assert f(hd=96) == EUNSUP and f(hd=256) == EUNSUP
    assert f(heads=0) == EINVAL and f(Tt=-1) == EINVAL
    assert f(st=Hh * 128) == OK            # contiguous q/k/v views of separate width
    assert f(st=Hh * 128 - 8) == EINVAL     # stride shorter than a row
    assert f(st=S + 4) == EALIGN
    assert f(qt=QT + 8) == EALIGN
    assert f(eps_t=-1.0) == EINVAL
    assert f(qo=KO) == EALIAS               # outputs overlap each other
    assert f(vo=QI + 64) == EALIAS          # output over an input
    assert f(Tt=0, qt=None) == OK           # an empty text stream may pass NULL
    assert f(Tt=0, Ti=0, qt=None, qi=None) == OK
    assert f(hd=64) == OK                  # head_dim 64: rows of 24 x 64 fit the same strides


def test_qk_neox_validation_matches(lib):
    QT, QI, WT, RT, RI, QO, KO, VO = (0x10000000 + i * 256 * MB for i in range(8))
    for hd, heads in ((128, 24), (64, 48)):
        S = 3 * heads * hd
        w = heads * hd * 2
        args = (QT, QT + w, QT + 2 * w, 256, S, QI, QI + w, QI + 2 * w, 4096, S, heads, hd,
                WT, WT + 256, WT + 512, WT + 768, RT, RI, EPS, EPS, QO, KO, VO)
        assert lib.dan_can_use_qk_norm_rope_neox_epilogue(*args) == OK
        assert lib.dan_can_use_qk_norm_rope_epilogue(*args) == OK
    bad = (QT, QT, QT, 1, 128, None, None, None, 0, 0, 1, 32, WT, WT, WT, WT, RT, RI, EPS, EPS,
           QO, KO, VO)
    assert lib.dan_can_use_qk_norm_rope_neox_epilogue(*bad) == EUNSUP


def test_binding_raises_without_cuda_tensors():
    import torch
    with pytest.raises(TypeError):
        ops.rms_modulate(torch.zeros(1, 2, 2048, dtype=torch.bfloat16),
                         torch.zeros(1, 2048, dtype=torch.bfloat16),
                         torch.zeros(1, 2048, dtype=torch.bfloat16), 1e-6)


def test_selftest_argument_checks(lib):
    # invalid limits are rejected before any CUDA call
    assert lib.dan_selftest_wait_timeout(0, None) == EINVAL
    assert lib.dan_selftest_wait_timeout(3_000_000_000, None) == EINVAL
    assert lib.dan_get_device_status(None) == EINVAL


def test_build_lists_every_source_and_header():
    """Every CUDA translation unit under csrc/ is compiled into libdan.so, and
    every header is a dependency of the rebuild check (a file missing from
    either list would be silently left out of the library or of the check)."""
    files = os.listdir(dan_build.CSRC)
    assert sorted(f for f in files if f.endswith(".cu")) == sorted(dan_build.SOURCES)
    assert sorted(f for f in files if f.endswith((".cuh", ".h"))) == sorted(dan_build.HEADERS)
