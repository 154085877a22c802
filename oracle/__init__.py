"""CPU oracle for the fused adaLN norm+modulate kernels -- TEST INFRASTRUCTURE.

Only the tests, ``__graft_entry__.smoke()`` and the bench's CPU-baseline leg
may import this package.  The product path (``dit_adaln_norm_gb300``) never
imports it and shares no code with it.

The arithmetic lives in ``oracle.c`` (plain C, every fp32 operation one IEEE
round-to-nearest step, contraction off); this module only compiles it and
marshals numpy arrays.  bf16 tensors travel as ``np.uint16`` bit patterns.

Parity status of each function (what pins it is in ``tests/test_oracle_pins.py``):

* ``round_bf16``: pinned (independent nearest-neighbour formulation in fp64).
* ``rms_modulate`` / ``gated_rms_modulate``: pinned (closed forms, +-a rows where
  eps matters, order probes with hand-derived sums, the weight product order and
  the division s/D at a width that is not a power of two worked by hand, fp64
  brute force within 2 bf16 ULP / 1e-6 rstd).
* ``ln_modulate``: pinned (constant rows, +-a rows, two- and three-chain combines
  worked by hand, the shfl.down lane and cross-warp orders, the combine's m2
  count weighting, product order and operand order worked by hand, exact 2^k
  scaling and sign symmetry, fp64 brute force).  The combine's parenthesisation
  and the cross-warp order are this library's reading of the pages; the
  hand-worked rows fix each of them.
* ``qk_norm_rope_epilogue``: pinned (cos=1/sin=0 and cos=0/sin=1 rotations,
  V copy, joint order, the head fold and the weight association worked by
  hand, eps per stream on small heads, fp64 brute force); with head_dim 64 and the neox
  rotation: the same closed forms, the neox rotation as a column
  permutation of the interleaved one, fp64 brute force.
* ``gated_ln_modulate``: pinned (r' against an independent elementwise
  formula, gate = 0 and the composition with ``ln_modulate`` of r').
* ``gated_residual_transposed``: pinned (torch bf16 ops on the transposed
  update, gate = 0 and gate = 1).
* ``fp8_e4m3``: pinned (every finite code decodes and re-encodes to itself,
  midpoints round to the even code, saturation, torch's float8_e4m3fn cast
  on the finite range, brute-force nearest code).
* ``ln_modulate_fp8``: pinned (elementwise equal to ``fp8_e4m3`` of
  ``ln_modulate`` times rn(1/qscale); constant rows give e4m3(shift/qscale)).
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_LIB = os.path.join(_HERE, "liboracle.so")

CFLAGS = ["-O2", "-std=c11", "-ffp-contract=off", "-fno-fast-math",
          "-fexcess-precision=standard", "-fPIC", "-shared"]


def build(force: bool = False) -> str:
    """Compile oracle.c into liboracle.so beside it (gcc, no GPU needed)."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + ".tmp%d" % os.getpid()
        subprocess.check_call(["gcc", *CFLAGS, "-o", tmp, _SRC, "-lm"])
        os.replace(tmp, _LIB)
    return _LIB


_lib = None
_P = ctypes.c_void_p
_I = ctypes.c_int64
_F = ctypes.c_float


def _load():
    global _lib
    if _lib is None:
        lib = ctypes.CDLL(build())
        lib.oracle_round_bf16.argtypes = [_P, _P, _I]
        lib.oracle_fp8_e4m3.argtypes = [_P, _P, _I]
        lib.oracle_gated_residual_transposed.argtypes = [_P, _P, _P, _I, _P, _I, _I, _I]
        lib.oracle_gated_ln_modulate.argtypes = [_P, _P, _P, _P, _P, _I, _P, _P, _I, _I, _I, _F,
                                                 _P]
        lib.oracle_ln_modulate_fp8.argtypes = [_P, _P, _P, _I, _F, _P, _I, _I, _I, _F]
        lib.oracle_rms_modulate.argtypes = [_P, _P, _P, _P, _I, _P, _I, _I, _I, _F, _P]
        lib.oracle_gated_rms_modulate.argtypes = [_P, _P, _P, _P, _P, _P, _I, _P, _P,
                                                  _I, _I, _I, _F, _P]
        lib.oracle_ln_modulate.argtypes = [_P, _P, _P, _I, _P, _I, _I, _I, _F, _P]
        lib.oracle_qk_norm_rope_epilogue.argtypes = (
            [_P, _P, _P, _I, _I] + [_P, _P, _P, _I, _I] + [_I] + [_P] * 4 + [_P, _P]
            + [_F, _F] + [_P, _P, _P, _P])
        lib.oracle_qk_norm_rope.argtypes = (
            [_P, _P, _P, _I, _I] + [_P, _P, _P, _I, _I] + [_I, ctypes.c_int, ctypes.c_int]
            + [_P] * 4 + [_P, _P] + [_F, _F] + [_P, _P, _P, _P])
        for f in ("oracle_round_bf16", "oracle_rms_modulate", "oracle_gated_rms_modulate",
                  "oracle_ln_modulate", "oracle_qk_norm_rope_epilogue"):
            getattr(lib, f).restype = None
        _lib = lib
    return _lib


def _ptr(a):
    return None if a is None else a.ctypes.data


def _bits(a, name):
    a = np.asarray(a)
    if a.dtype != np.uint16:
        raise TypeError(f"{name}: expected uint16 bf16 bit patterns, got {a.dtype}")
    return a


def _rows(x, name):
    """Contiguous [B, T, D] bf16 bits."""
    x = np.ascontiguousarray(_bits(x, name))
    if x.ndim != 3:
        raise ValueError(f"{name}: expected [B, T, D]")
    return x


def _vec(v, B, D, name):
    """A [B, D] view whose rows may be strided (e.g. chunks of an embedding);
    returns (array to pass, batch stride in elements)."""
    v = _bits(v, name)
    if v.ndim == 1:
        v = v[None, :]
    if v.shape != (B, D) or v.strides[1] != 2 or v.strides[0] % 2:
        raise ValueError(f"{name}: expected a [B={B}, D={D}] view with unit column stride")
    return v, v.strides[0] // 2


def _vec_stride(vecs):
    strides = {s for _, s in vecs}
    if len(strides) != 1:
        raise ValueError("all per-batch vectors must share one batch stride")
    return strides.pop()


def round_bf16(f32):
    f32 = np.ascontiguousarray(f32, dtype=np.float32)
    out = np.empty(f32.shape, np.uint16)
    _load().oracle_round_bf16(_ptr(f32), _ptr(out), f32.size)
    return out


def rms_modulate(x, scale, shift, eps, weight=None, with_stats=False):
    x = _rows(x, "x")
    B, T, D = x.shape
    if D % 64:
        raise ValueError("RMS oracle needs D % 64 == 0")
    sc, ss = _vec(scale, B, D, "scale")
    sh, hs = _vec(shift, B, D, "shift")
    vs = _vec_stride([(sc, ss), (sh, hs)])
    w = None if weight is None else np.ascontiguousarray(_bits(weight, "weight"))
    y = np.empty_like(x)
    st = np.empty((B * T, 2), np.float32) if with_stats else None
    _load().oracle_rms_modulate(_ptr(x), _ptr(w), _ptr(sc), _ptr(sh), vs, _ptr(y),
                                B, T, D, float(eps), _ptr(st))
    return (y, st) if with_stats else y


def gated_rms_modulate(r, h, gate, scale, shift, eps, weight=None, with_stats=False):
    r = _rows(r, "r")
    h = _rows(h, "h")
    B, T, D = r.shape
    if h.shape != r.shape or D % 64:
        raise ValueError("gated oracle: r, h must match and D % 64 == 0")
    g, gs = _vec(gate, B, D, "gate")
    sc, ss = _vec(scale, B, D, "scale")
    sh, hs = _vec(shift, B, D, "shift")
    vs = _vec_stride([(g, gs), (sc, ss), (sh, hs)])
    w = None if weight is None else np.ascontiguousarray(_bits(weight, "weight"))
    r_out = np.empty_like(r)
    y = np.empty_like(r)
    st = np.empty((B * T, 2), np.float32) if with_stats else None
    _load().oracle_gated_rms_modulate(_ptr(r), _ptr(h), _ptr(g), _ptr(w), _ptr(sc), _ptr(sh),
                                      vs, _ptr(r_out), _ptr(y), B, T, D, float(eps), _ptr(st))
    return (r_out, y, st) if with_stats else (r_out, y)


def ln_modulate(x, scale, shift, eps, with_stats=False):
    x = _rows(x, "x")
    B, T, D = x.shape
    if D % 8:
        raise ValueError("LayerNorm oracle needs D % 8 == 0")
    sc, ss = _vec(scale, B, D, "scale")
    sh, hs = _vec(shift, B, D, "shift")
    vs = _vec_stride([(sc, ss), (sh, hs)])
    y = np.empty_like(x)
    st = np.empty((B * T, 3), np.float32) if with_stats else None
    _load().oracle_ln_modulate(_ptr(x), _ptr(sc), _ptr(sh), vs, _ptr(y), B, T, D,
                               float(eps), _ptr(st))
    return (y, st) if with_stats else y


def _qkv_views(q, k, v, name):
    """q, k, v: [T, H*head_dim] views sharing one row stride (unit column stride)."""
    arrs = [_bits(a, f"{name}.{n}") for a, n in zip((q, k, v), "qkv")]
    T, HD = arrs[0].shape
    if T == 0:  # an empty stream: nothing is read, strides are irrelevant
        return [np.zeros((0, HD), np.uint16)] * 3, 0, HD, HD
    for a in arrs:
        if a.shape != (T, HD) or a.strides[1] != 2:
            raise ValueError(f"{name}: q, k, v must be [T, H*head_dim] views, unit column stride")
    strides = {a.strides[0] // 2 for a in arrs}
    if len(strides) != 1:
        raise ValueError(f"{name}: q, k, v must share one row stride")
    return arrs, T, HD, strides.pop()


def qk_norm_rope_epilogue(txt, img, H, weights, rope_txt, rope_img, eps_txt, eps_img,
                          with_stats=False, head_dim=128, neox=False):
    """txt, img: (q, k, v) views [T_s, H*head_dim]; weights: (wq_txt, wk_txt,
    wq_img, wk_img) [head_dim] bf16; rope_*: fp32 [T_s, head_dim].  Returns
    joint q, k, v as [T_txt + T_img, H, head_dim] (and rstd [T, 2, H] if
    with_stats).  head_dim 128 or 64; neox rotates (i, i + head_dim/2)
    instead of interleaved pairs."""
    if head_dim not in (64, 128):
        raise ValueError("head_dim must be 64 or 128")
    (qt, kt, vt), Tt, HDt, st_ = _qkv_views(*txt, "txt")
    (qi, ki, vi), Ti, HDi, si_ = _qkv_views(*img, "img")
    if HDt != H * head_dim or HDi != H * head_dim:
        raise ValueError("q, k, v must be [T, H*head_dim]")
    ws = [np.ascontiguousarray(_bits(w, "weight")) for w in weights]
    rt = np.ascontiguousarray(rope_txt, dtype=np.float32)
    ri = np.ascontiguousarray(rope_img, dtype=np.float32)
    if rt.shape != (Tt, head_dim) or ri.shape != (Ti, head_dim):
        raise ValueError("rope tables must be [T_s, head_dim] fp32")
    T = Tt + Ti
    qo = np.empty((T, H, head_dim), np.uint16)
    ko = np.empty_like(qo)
    vo = np.empty_like(qo)
    rs = np.empty((T, 2, H), np.float32) if with_stats else None
    _load().oracle_qk_norm_rope(
        _ptr(qt), _ptr(kt), _ptr(vt), Tt, st_, _ptr(qi), _ptr(ki), _ptr(vi), Ti, si_, H,
        head_dim, int(bool(neox)), *[_ptr(w) for w in ws], _ptr(rt), _ptr(ri), float(eps_txt),
        float(eps_img), _ptr(qo), _ptr(ko), _ptr(vo), _ptr(rs))
    return (qo, ko, vo, rs) if with_stats else (qo, ko, vo)


def fp8_e4m3(values):
    """fp32 values -> E4M3 codes (uint8): nearest, ties to even, saturated
    to +-448; NaN -> 0x7F."""
    v = np.ascontiguousarray(values, dtype=np.float32)
    out = np.empty(v.shape, np.uint8)
    _load().oracle_fp8_e4m3(_ptr(v), _ptr(out), v.size)
    return out


def ln_modulate_fp8(x, scale, shift, qscale, eps):
    """E4M3 codes of ln_modulate(x, scale, shift, eps) * rn(1/qscale)."""
    x = _rows(x, "x")
    B, T, D = x.shape
    if D % 8:
        raise ValueError("LayerNorm oracle needs D % 8 == 0")
    if not (np.isfinite(qscale) and qscale > 0):
        raise ValueError("qscale must be finite and > 0")
    sc, ss = _vec(scale, B, D, "scale")
    sh, hs = _vec(shift, B, D, "shift")
    vs = _vec_stride([(sc, ss), (sh, hs)])
    q = np.empty((B, T, D), np.uint8)
    _load().oracle_ln_modulate_fp8(_ptr(x), _ptr(sc), _ptr(sh), vs, float(qscale), _ptr(q),
                                   B, T, D, float(eps))
    return q


def gated_ln_modulate(r, h, gate, scale, shift, eps, with_stats=False):
    """r' = bf16(r + bf16(gate * h)); y = ln_modulate(r').  Returns (r', y)."""
    r = _rows(r, "r")
    h = _rows(h, "h")
    B, T, D = r.shape
    if h.shape != r.shape or D % 8:
        raise ValueError("gated LayerNorm oracle: r, h must match and D % 8 == 0")
    g, gs = _vec(gate, B, D, "gate")
    sc, ss = _vec(scale, B, D, "scale")
    sh, hs = _vec(shift, B, D, "shift")
    vs = _vec_stride([(g, gs), (sc, ss), (sh, hs)])
    r_out = np.empty_like(r)
    y = np.empty_like(r)
    st = np.empty((B * T, 3), np.float32) if with_stats else None
    _load().oracle_gated_ln_modulate(_ptr(r), _ptr(h), _ptr(g), _ptr(sc), _ptr(sh), vs,
                                     _ptr(r_out), _ptr(y), B, T, D, float(eps), _ptr(st))
    return (r_out, y, st) if with_stats else (r_out, y)


def gated_residual_transposed(r, h, gate):
    """r, h: the residual [B, D, T] and the update [B, T, D] (bf16 bits);
    gate [B, D].  Returns r' = bf16(r + bf16(gate * h^T)) as [B, D, T]."""
    r = _rows(r, "r")
    h = _rows(h, "h")
    B, D, T = r.shape
    if h.shape != (B, T, D):
        raise ValueError("h must be [B, T, D] for a residual [B, D, T]")
    g, gs = _vec(gate, B, D, "gate")
    vs = _vec_stride([(g, gs)])
    out = np.empty_like(r)
    _load().oracle_gated_residual_transposed(_ptr(r), _ptr(h), _ptr(g), vs, _ptr(out), B, T, D)
    return out
