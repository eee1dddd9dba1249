"""fp64 CPU oracle for grouped 2D convolution (NCHW) -- TEST INFRASTRUCTURE ONLY.

This package is the parity oracle for the CUDA library in ``bwd_gconv_fwd_gb300``.
It shares no code with that library and the library never imports it.  Only
``tests/``, ``__graft_entry__.smoke()`` and ``bench.py``'s CPU-baseline leg use it.

The arithmetic lives in ``gconv_oracle.c`` (plain direct loops in fp64, one
defining sum per output element); this module compiles it with gcc and wraps it
with ctypes.  Inputs are float64 numpy arrays in NCHW / [C_out, C_in/G, kH, kW]
layout; geometry is the 14-tuple
``(N, C_in, H, W, C_out, kH, kW, stride, pad_top, pad_bottom, pad_left, pad_right,
dilation, groups)`` (stride and dilation the same on both axes) or the 16-tuple
``(N, C_in, H, W, C_out, kH, kW, stride_h, stride_w, pad_top, pad_bottom, pad_left,
pad_right, dilation_h, dilation_w, groups)``.

Parity status: every entry point is pinned in ``tests/test_oracle.py`` against
brute force, library routines (scipy correlate2d, numpy matmul, torch conv2d in
float64 with autograd), the adjoint identities, finite differences, closed forms
of the all-ones fully-connected-mode script and shape arithmetic.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import sys

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "gconv_oracle.c")
_LIB_PATH = os.path.join(_HERE, "liboracle.so")
_lib = None

GEOM_FIELDS = ("N", "C_in", "H", "W", "C_out", "kH", "kW", "stride_h", "stride_w",
               "pad_top", "pad_bottom", "pad_left", "pad_right", "dilation_h", "dilation_w", "groups")


def geom16(g):
    """The 16-integer geometry of a 14- or 16-tuple (a 14-tuple has one stride and one
    dilation for both axes)."""
    g = tuple(int(v) for v in g)
    if len(g) == 14:
        N, Cin, H, W, Cout, kH, kW, s, pt, pb, pl, pr, d, G = g
        return (N, Cin, H, W, Cout, kH, kW, s, s, pt, pb, pl, pr, d, d, G)
    if len(g) == 16:
        return g
    raise ValueError("geometry must have 14 or 16 integers")


def build(force: bool = False) -> str:
    """Compile the oracle shared library with gcc (-O2, OpenMP) if needed."""
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-fopenmp", "-fPIC", "-shared", "-std=c99", _SRC, "-o", tmp, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    if _lib is not None:
        return _lib
    build()
    lib = ctypes.CDLL(_LIB_PATH)
    P = ctypes.POINTER
    dp = P(ctypes.c_double)
    ip = P(ctypes.c_int)
    i64 = ctypes.c_int64
    i64p = P(ctypes.c_int64)
    lib.oracle_out_shape.argtypes = [ip, ip, ip]
    lib.oracle_fwd.argtypes = [ip, dp, dp, dp, dp, ctypes.c_int]
    lib.oracle_bwd_data.argtypes = [ip, dp, dp, dp, ctypes.c_int]
    lib.oracle_bwd_weight.argtypes = [ip, dp, dp, dp, ctypes.c_int]
    lib.oracle_bwd_bias.argtypes = [ip, dp, dp, ctypes.c_int]
    lib.oracle_fwd_points.argtypes = [ip, dp, dp, dp, i64, i64p, dp, ctypes.c_int]
    lib.oracle_bwd_data_points.argtypes = [ip, dp, dp, i64, i64p, dp, ctypes.c_int]
    lib.oracle_bwd_weight_points.argtypes = [ip, dp, dp, i64, i64p, dp, ctypes.c_int]
    lib.oracle_max_threads.argtypes = []
    for name in ("oracle_out_shape", "oracle_fwd", "oracle_bwd_data", "oracle_bwd_weight",
                 "oracle_bwd_bias", "oracle_fwd_points", "oracle_bwd_data_points",
                 "oracle_bwd_weight_points", "oracle_max_threads"):
        getattr(lib, name).restype = ctypes.c_int
    _lib = lib
    return lib


def _geom(g) -> ctypes.Array:
    return (ctypes.c_int * 16)(*geom16(g))


def _dptr(a):
    if a is None:
        return None
    return a.ctypes.data_as(ctypes.POINTER(ctypes.c_double))


def _f64(a, shape, name):
    a = np.ascontiguousarray(np.asarray(a, dtype=np.float64))
    if tuple(a.shape) != tuple(shape):
        raise ValueError(f"{name}: shape {a.shape} != {shape}")
    return a


def out_shape(g):
    """(Ho, Wo) for geometry g, or ValueError if the geometry is malformed."""
    ho, wo = ctypes.c_int(), ctypes.c_int()
    if _load().oracle_out_shape(_geom(g), ctypes.byref(ho), ctypes.byref(wo)):
        raise ValueError(f"invalid geometry {tuple(g)}")
    return ho.value, wo.value


def shapes(g):
    """Shapes of x, w, b, y for geometry g."""
    N, Cin, H, W, Cout, kH, kW, sh, sw, pt, pb, pl, pr, dh, dw, G = geom16(g)
    Ho, Wo = out_shape(g)
    return dict(x=(N, Cin, H, W), w=(Cout, Cin // G, kH, kW), b=(Cout,), y=(N, Cout, Ho, Wo))


def max_threads() -> int:
    return int(_load().oracle_max_threads())


def fwd(g, x, w, b=None, threads: int = 0):
    sh = shapes(g)
    x, w = _f64(x, sh["x"], "x"), _f64(w, sh["w"], "w")
    b = None if b is None else _f64(b, sh["b"], "b")
    y = np.empty(sh["y"], np.float64)
    if _load().oracle_fwd(_geom(g), _dptr(x), _dptr(w), _dptr(b), _dptr(y), threads):
        raise ValueError("oracle_fwd rejected the geometry")
    return y


def bwd_data(g, dy, w, threads: int = 0):
    sh = shapes(g)
    dy, w = _f64(dy, sh["y"], "dy"), _f64(w, sh["w"], "w")
    dx = np.empty(sh["x"], np.float64)
    if _load().oracle_bwd_data(_geom(g), _dptr(dy), _dptr(w), _dptr(dx), threads):
        raise ValueError("oracle_bwd_data rejected the geometry")
    return dx


def bwd_weight(g, x, dy, threads: int = 0):
    sh = shapes(g)
    x, dy = _f64(x, sh["x"], "x"), _f64(dy, sh["y"], "dy")
    dw = np.empty(sh["w"], np.float64)
    if _load().oracle_bwd_weight(_geom(g), _dptr(x), _dptr(dy), _dptr(dw), threads):
        raise ValueError("oracle_bwd_weight rejected the geometry")
    return dw


def bwd_bias(g, dy, threads: int = 0):
    sh = shapes(g)
    dy = _f64(dy, sh["y"], "dy")
    db = np.empty(sh["b"], np.float64)
    if _load().oracle_bwd_bias(_geom(g), _dptr(dy), _dptr(db), threads):
        raise ValueError("oracle_bwd_bias rejected the geometry")
    return db


def _idx(idx):
    idx = np.ascontiguousarray(np.asarray(idx, dtype=np.int64).ravel())
    return idx, idx.ctypes.data_as(ctypes.POINTER(ctypes.c_int64))


def fwd_points(g, x, w, b, flat_idx, threads: int = 0):
    """y at the given flat NCHW indices."""
    sh = shapes(g)
    x, w = _f64(x, sh["x"], "x"), _f64(w, sh["w"], "w")
    b = None if b is None else _f64(b, sh["b"], "b")
    idx, ip = _idx(flat_idx)
    if idx.size and (idx.min() < 0 or idx.max() >= int(np.prod(sh["y"]))):
        raise IndexError("flat index out of range")
    out = np.empty(idx.size, np.float64)
    _load().oracle_fwd_points(_geom(g), _dptr(x), _dptr(w), _dptr(b), idx.size, ip, _dptr(out), threads)
    return out


def bwd_data_points(g, dy, w, flat_idx, threads: int = 0):
    """dx at the given flat NCHW indices."""
    sh = shapes(g)
    dy, w = _f64(dy, sh["y"], "dy"), _f64(w, sh["w"], "w")
    idx, ip = _idx(flat_idx)
    if idx.size and (idx.min() < 0 or idx.max() >= int(np.prod(sh["x"]))):
        raise IndexError("flat index out of range")
    out = np.empty(idx.size, np.float64)
    _load().oracle_bwd_data_points(_geom(g), _dptr(dy), _dptr(w), idx.size, ip, _dptr(out), threads)
    return out


def bwd_weight_points(g, x, dy, flat_idx, threads: int = 0):
    """dw at the given flat [C_out, C_in/G, kH, kW] indices."""
    sh = shapes(g)
    x, dy = _f64(x, sh["x"], "x"), _f64(dy, sh["y"], "dy")
    idx, ip = _idx(flat_idx)
    if idx.size and (idx.min() < 0 or idx.max() >= int(np.prod(sh["w"]))):
        raise IndexError("flat index out of range")
    out = np.empty(idx.size, np.float64)
    _load().oracle_bwd_weight_points(_geom(g), _dptr(x), _dptr(dy), idx.size, ip, _dptr(out), threads)
    return out


if __name__ == "__main__":  # pragma: no cover
    print(build(force="--force" in sys.argv))
