"""Thin ctypes binding of libdan.so (include/dan.h): argument marshalling only.

Every function takes CUDA bf16 torch tensors, checks the layout the C ABI
expects, passes raw pointers, strides and the current CUDA stream, and turns
a non-zero status into an exception.  All arithmetic runs in the CUDA
kernels; there is no CPU or eager fallback.  PyTorch only allocates outputs.

The library is loaded on first use.  If it is missing the call raises
(build it with ``python -c "import __graft_entry__ as g; g.build()"``).
"""
from __future__ import annotations

import ctypes
import os
import re

import torch

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "libdan.so")
HEADER = os.path.join(os.path.dirname(HERE), "include", "dan.h")

DAN_OK, DAN_EINVAL, DAN_EUNSUPPORTED, DAN_EALIGN, DAN_EALIAS, DAN_ECUDA = range(6)

_P = ctypes.c_void_p
_I = ctypes.c_int64
_F = ctypes.c_float
_SIGS = {
    "dan_rms_modulate": [_P, _P, _P, _P, _I, _P, _I, _I, _I, _F, _P],
    "dan_rms_modulate_noalloc": [_P, _P, _P, _P, _I, _P, _I, _I, _I, _F, _P],
    "dan_can_use_rms_modulate": [_P, _P, _P, _P, _I, _P, _I, _I, _I, _F],
    "dan_gated_rms_modulate": [_P, _P, _P, _P, _P, _P, _I, _P, _P, _I, _I, _I, _F, _P],
    "dan_can_use_gated_rms_modulate": [_P, _P, _P, _P, _P, _P, _I, _P, _P, _I, _I, _I, _F],
    "dan_ln_modulate": [_P, _P, _P, _I, _P, _I, _I, _I, _F, _P],
    "dan_can_use_ln_modulate": [_P, _P, _P, _I, _P, _I, _I, _I, _F],
    "dan_ln_modulate_fp8": [_P, _P, _P, _I, _F, _P, _I, _I, _I, _F, _P],
    "dan_gated_residual_transposed": [_P, _P, _P, _I, _P, _I, _I, _I, _P],
    "dan_can_use_gated_residual_transposed": [_P, _P, _P, _I, _P, _I, _I, _I],
    "dan_gated_ln_modulate": [_P, _P, _P, _P, _P, _I, _P, _P, _I, _I, _I, _F, _P],
    "dan_can_use_gated_ln_modulate": [_P, _P, _P, _P, _P, _I, _P, _P, _I, _I, _I, _F],
    "dan_can_use_ln_modulate_fp8": [_P, _P, _P, _I, _F, _P, _I, _I, _I, _F],
    "dan_qk_norm_rope_epilogue": [_P, _P, _P, _I, _I, _P, _P, _P, _I, _I, _I, _I,
                                  _P, _P, _P, _P, _P, _P, _F, _F, _P, _P, _P, _P],
    "dan_can_use_qk_norm_rope_epilogue": [_P, _P, _P, _I, _I, _P, _P, _P, _I, _I, _I, _I,
                                          _P, _P, _P, _P, _P, _P, _F, _F, _P, _P, _P],
    "dan_qk_norm_rope_neox_epilogue": [_P, _P, _P, _I, _I, _P, _P, _P, _I, _I, _I, _I,
                                       _P, _P, _P, _P, _P, _P, _F, _F, _P, _P, _P, _P],
    "dan_can_use_qk_norm_rope_neox_epilogue": [_P, _P, _P, _I, _I, _P, _P, _P, _I, _I, _I, _I,
                                               _P, _P, _P, _P, _P, _P, _F, _F, _P, _P, _P],
}

_lib = None


class DanError(RuntimeError):
    def __init__(self, status: int, what: str):
        self.status = status
        super().__init__(f"{what}: {status_string(status)}")


def load():
    """Load libdan.so (raises if it was not built)."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"libdan.so not found at {LIB_PATH}: build the CUDA library first")
        lib = ctypes.CDLL(LIB_PATH)
        for name, args in _SIGS.items():
            fn = getattr(lib, name)
            fn.argtypes = args
            fn.restype = ctypes.c_int
        lib.dan_status_string.argtypes = [ctypes.c_int]
        lib.dan_status_string.restype = ctypes.c_char_p
        lib.dan_get_device_status.argtypes = [ctypes.POINTER(ctypes.c_uint)]
        lib.dan_get_device_status.restype = ctypes.c_int
        lib.dan_selftest_wait_timeout.argtypes = [ctypes.c_ulonglong, _P]
        lib.dan_selftest_wait_timeout.restype = ctypes.c_int
        _lib = lib
    return _lib


def declared_symbols() -> list[str]:
    """Function names declared in include/dan.h."""
    text = open(HEADER).read()
    return sorted(set(re.findall(r"\b(dan_\w+)\s*\(", text)))


def status_string(status: int) -> str:
    return load().dan_status_string(int(status)).decode()


def device_status() -> int:
    """Read and clear the current device's status word (bit 1: a warp gave
    up waiting for a row it requested, 4: it then also gave up on its other
    copies in flight).  Synchronous; 0 when every wait completed."""
    v = ctypes.c_uint(0)
    _check(load().dan_get_device_status(ctypes.byref(v)), "dan_get_device_status")
    return v.value


def selftest_wait_timeout(limit_ns: int):
    """Launch the bounded-wait self-test on the current stream."""
    _check(load().dan_selftest_wait_timeout(int(limit_ns), _stream()), "dan_selftest_wait_timeout")


def _stream() -> int:
    return torch.cuda.current_stream().cuda_stream


def _check(status: int, what: str):
    if status != DAN_OK:
        raise DanError(status, what)


def _bf16_cuda(t: torch.Tensor, name: str):
    if not isinstance(t, torch.Tensor) or not t.is_cuda or t.dtype != torch.bfloat16:
        raise TypeError(f"{name}: expected a CUDA bfloat16 tensor")


def _ptr(t):
    return None if t is None else t.data_ptr()


def _rows(x: torch.Tensor, name: str):
    _bf16_cuda(x, name)
    if x.dim() != 3 or not x.is_contiguous():
        raise ValueError(f"{name}: expected a contiguous [B, T, D] tensor")
    return x.shape


def _vectors(B: int, D: int, named):
    """Per-batch [B, D] (or [D] when B == 1) views sharing one batch stride."""
    strides = set()
    for name, v in named:
        _bf16_cuda(v, name)
        if v.dim() == 1:
            if B != 1 or v.shape[0] != D or v.stride(0) != 1:
                raise ValueError(f"{name}: a 1-D vector needs B == 1, shape [D], unit stride")
            strides.add(None)
            continue
        if tuple(v.shape) != (B, D) or v.stride(1) != 1:
            raise ValueError(f"{name}: expected a [B={B}, D={D}] view with unit column stride")
        strides.add(v.stride(0) if B > 1 else None)
    strides.discard(None)
    if len(strides) > 1:
        raise ValueError("per-batch vectors must share one batch stride")
    return strides.pop() if strides else D


def _weight(w, D):
    if w is None:
        return None
    _bf16_cuda(w, "weight")
    if w.dim() != 1 or w.shape[0] != D or not w.is_contiguous():
        raise ValueError("weight: expected a contiguous [D] tensor")
    return w


def rms_modulate(x, scale, shift, eps: float, weight=None, out=None):
    """y = bf16(RMSNorm(x) [* weight] * (1 + scale) + shift), x [B, T, D]."""
    B, T, D = _rows(x, "x")
    vs = _vectors(B, D, [("scale", scale), ("shift", shift)])
    weight = _weight(weight, D)
    y = torch.empty_like(x) if out is None else out
    _rows(y, "out")
    _check(load().dan_rms_modulate(_ptr(x), _ptr(weight), _ptr(scale), _ptr(shift), vs, _ptr(y),
                                   B, T, D, float(eps), _stream()), "dan_rms_modulate")
    return y


def gated_rms_modulate(r, h, gate, scale, shift, eps: float, weight=None, r_out=None, out=None):
    """r' = bf16(r + bf16(gate * h)); y = rms_modulate(r').  Returns (r', y)."""
    B, T, D = _rows(r, "r")
    _rows(h, "h")
    vs = _vectors(B, D, [("gate", gate), ("scale", scale), ("shift", shift)])
    weight = _weight(weight, D)
    r_out = torch.empty_like(r) if r_out is None else r_out
    y = torch.empty_like(r) if out is None else out
    _rows(r_out, "r_out")
    _rows(y, "out")
    _check(load().dan_gated_rms_modulate(_ptr(r), _ptr(h), _ptr(gate), _ptr(weight), _ptr(scale),
                                         _ptr(shift), vs, _ptr(r_out), _ptr(y), B, T, D,
                                         float(eps), _stream()), "dan_gated_rms_modulate")
    return r_out, y


def ln_modulate(x, scale, shift, eps: float, out=None):
    """y = bf16(LayerNorm(x) * (1 + scale) + shift), LayerNorm without affine."""
    B, T, D = _rows(x, "x")
    vs = _vectors(B, D, [("scale", scale), ("shift", shift)])
    y = torch.empty_like(x) if out is None else out
    _rows(y, "out")
    _check(load().dan_ln_modulate(_ptr(x), _ptr(scale), _ptr(shift), vs, _ptr(y), B, T, D,
                                  float(eps), _stream()), "dan_ln_modulate")
    return y


def gated_ln_modulate(r, h, gate, scale, shift, eps: float, r_out=None, out=None):
    """r' = bf16(r + bf16(gate * h)); y = ln_modulate(r').  Returns (r', y)."""
    B, T, D = _rows(r, "r")
    _rows(h, "h")
    vs = _vectors(B, D, [("gate", gate), ("scale", scale), ("shift", shift)])
    r_out = torch.empty_like(r) if r_out is None else r_out
    y = torch.empty_like(r) if out is None else out
    _rows(r_out, "r_out")
    _rows(y, "out")
    _check(load().dan_gated_ln_modulate(_ptr(r), _ptr(h), _ptr(gate), _ptr(scale), _ptr(shift),
                                        vs, _ptr(r_out), _ptr(y), B, T, D, float(eps),
                                        _stream()), "dan_gated_ln_modulate")
    return r_out, y


def gated_residual_transposed(r, h, gate, out=None):
    """r: the residual [B, D, T] (the [B, hidden, tokens] layout); h: the
    update [B, T, D]; gate [B, D] (or [D] when B == 1).  Returns
    r' = bf16(r + bf16(gate * h^T)) as [B, D, T]."""
    _bf16_cuda(r, "r")
    _bf16_cuda(h, "h")
    if r.dim() != 3 or not r.is_contiguous():
        raise ValueError("r: expected a contiguous [B, D, T] tensor")
    B, D, T = r.shape
    if tuple(h.shape) != (B, T, D) or not h.is_contiguous():
        raise ValueError("h: expected a contiguous [B, T, D] tensor")
    vs = _vectors(B, D, [("gate", gate)])
    y = torch.empty_like(r) if out is None else out
    _bf16_cuda(y, "out")
    if tuple(y.shape) != (B, D, T) or not y.is_contiguous():
        raise ValueError("out: expected a contiguous [B, D, T] tensor")
    _check(load().dan_gated_residual_transposed(_ptr(r), _ptr(h), _ptr(gate), vs, _ptr(y), B, T,
                                                D, _stream()), "dan_gated_residual_transposed")
    return y


def ln_modulate_fp8(x, scale, shift, qscale: float, eps: float, out=None):
    """q = e4m3(ln_modulate(x, scale, shift, eps) * rn(1/qscale)) as a
    torch.uint8 [B, T, D] tensor of E4M3 codes (view it as
    torch.float8_e4m3fn for an FP8 GEMM)."""
    B, T, D = _rows(x, "x")
    vs = _vectors(B, D, [("scale", scale), ("shift", shift)])
    q = torch.empty((B, T, D), dtype=torch.uint8, device=x.device) if out is None else out
    if q.dtype != torch.uint8 or not q.is_cuda or tuple(q.shape) != (B, T, D) or not q.is_contiguous():
        raise ValueError("out: expected a contiguous CUDA uint8 [B, T, D] tensor")
    _check(load().dan_ln_modulate_fp8(_ptr(x), _ptr(scale), _ptr(shift), vs, float(qscale),
                                      _ptr(q), B, T, D, float(eps), _stream()),
           "dan_ln_modulate_fp8")
    return q


def _qkv(views, name, heads, hd):
    q, k, v = views
    T = q.shape[0]
    for t, n in zip(views, "qkv"):
        _bf16_cuda(t, f"{name}.{n}")
        if t.dim() != 2 or t.shape != (T, heads * hd) or (T > 0 and t.stride(1) != 1):
            raise ValueError(f"{name}.{n}: expected a [T, heads*{hd}] view with unit column stride")
    strides = {t.stride(0) for t in views} if T > 1 else {heads * hd}
    if len(strides) != 1:
        raise ValueError(f"{name}: q, k, v must share one row stride")
    return T, strides.pop()


def qk_norm_rope_epilogue(txt, img, wq_txt, wk_txt, wq_img, wk_img, rope_txt, rope_img,
                          eps_txt: float, eps_img: float, heads: int, out=None,
                          head_dim: int = 128, neox: bool = False):
    """txt, img: (q, k, v) views [T_s, heads*head_dim]; weights [head_dim] bf16;
    rope tables fp32 [T_s, head_dim].  Returns joint (q, k, v), each
    [T_txt+T_img, heads, head_dim].  head_dim 128 or 64; neox=True rotates
    the halves' pairs (dan_qk_norm_rope_neox_epilogue) instead of
    interleaved pairs."""
    hd = int(head_dim)
    Tt, st = _qkv(txt, "txt", heads, hd)
    Ti, si = _qkv(img, "img", heads, hd)
    for w, n in ((wq_txt, "wq_txt"), (wk_txt, "wk_txt"), (wq_img, "wq_img"), (wk_img, "wk_img")):
        _bf16_cuda(w, n)
        if w.shape != (hd,) or not w.is_contiguous():
            raise ValueError(f"{n}: expected a contiguous [{hd}] tensor")
    for r, n, T in ((rope_txt, "rope_txt", Tt), (rope_img, "rope_img", Ti)):
        if not r.is_cuda or r.dtype != torch.float32 or r.shape != (T, hd) or not r.is_contiguous():
            raise ValueError(f"{n}: expected a contiguous CUDA float32 [T, {hd}] tensor")
    if out is None:
        dev = txt[0].device
        out = tuple(torch.empty((Tt + Ti, heads, hd), dtype=torch.bfloat16, device=dev)
                    for _ in range(3))
    qo, ko, vo = out
    name = "dan_qk_norm_rope_neox_epilogue" if neox else "dan_qk_norm_rope_epilogue"
    _check(getattr(load(), name)(
        _ptr(txt[0]), _ptr(txt[1]), _ptr(txt[2]), Tt, st,
        _ptr(img[0]), _ptr(img[1]), _ptr(img[2]), Ti, si, heads, hd,
        _ptr(wq_txt), _ptr(wk_txt), _ptr(wq_img), _ptr(wk_img), _ptr(rope_txt), _ptr(rope_img),
        float(eps_txt), float(eps_img), _ptr(qo), _ptr(ko), _ptr(vo), _stream()), name)
    return qo, ko, vo
