"""ctypes wrapper of the plain C fp32 combine in ``combine_f32.c``.

Test infrastructure only (see the package docstring).  ``build()`` compiles
the C file with gcc into ``oracle/_combine_f32.so`` (no implicit FMA
contraction, no fast-math), and ``load()`` builds it on first use if missing.
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "combine_f32.c")
_LIB = os.path.join(_HERE, "_combine_f32.so")
_lib = None


def build(force: bool = False) -> str:
    if force or not os.path.exists(_LIB) or (
            os.path.getmtime(_LIB) < os.path.getmtime(_SRC)):
        cmd = ["gcc", "-O2", "-std=c11", "-shared", "-fPIC",
               "-ffp-contract=off", "-fno-fast-math", "-fno-builtin",
               "-o", _LIB + ".tmp", _SRC, "-lm"]
        subprocess.run(cmd, check=True)
        os.replace(_LIB + ".tmp", _LIB)
    return _LIB


def load():
    global _lib
    if _lib is None:
        lib = ctypes.CDLL(build())
        fp = ctypes.POINTER(ctypes.c_float)
        lib.fa_oracle_exp2f.argtypes = [ctypes.c_float]
        lib.fa_oracle_exp2f.restype = ctypes.c_float
        lib.fa_oracle_lnf.argtypes = [ctypes.c_float]
        lib.fa_oracle_lnf.restype = ctypes.c_float
        lib.fa_oracle_combine_f32.argtypes = [
            fp, fp, fp, ctypes.c_int, ctypes.c_int, ctypes.c_int, fp,
            ctypes.POINTER(ctypes.c_uint16), fp]
        lib.fa_oracle_combine_f32.restype = ctypes.c_int
        lib.fa_oracle_welford_combine_f32.argtypes = [
            fp, fp, fp, ctypes.c_int, ctypes.c_int, ctypes.c_float, fp, fp, fp]
        lib.fa_oracle_welford_combine_f32.restype = ctypes.c_int
        _lib = lib
    return _lib


def exp2f(x: float) -> float:
    return float(load().fa_oracle_exp2f(ctypes.c_float(x)))


def lnf(x: float) -> float:
    return float(load().fa_oracle_lnf(ctypes.c_float(x)))


def _fptr(a: np.ndarray):
    return a.ctypes.data_as(ctypes.POINTER(ctypes.c_float))


def combine_f32(part_m, part_d, part_o):
    """part_m, part_d [rows, S]; part_o [rows, S, D] (anything castable to
    float32; the cast must be exact for bit comparisons).  Returns
    (O fp32 [rows, D], O bf16 bits uint16 [rows, D], LSE fp32 [rows])."""
    m = np.ascontiguousarray(part_m, dtype=np.float32)
    d = np.ascontiguousarray(part_d, dtype=np.float32)
    o = np.ascontiguousarray(part_o, dtype=np.float32)
    rows, S = m.shape
    D = o.shape[-1]
    assert d.shape == (rows, S) and o.shape == (rows, S, D)
    out_o = np.empty((rows, D), np.float32)
    out_b = np.empty((rows, D), np.uint16)
    out_l = np.empty((rows,), np.float32)
    rc = load().fa_oracle_combine_f32(
        _fptr(m), _fptr(d), _fptr(o), rows, S, D, _fptr(out_o),
        out_b.ctypes.data_as(ctypes.POINTER(ctypes.c_uint16)), _fptr(out_l))
    if rc != 0:
        raise ValueError("fa_oracle_combine_f32: bad sizes")
    return out_o, out_b, out_l


def welford_combine_f32(part_n, part_mu, part_m2, eps=0.0):
    """part_* [rows, S] (castable exactly to float32).  Returns mean, var and
    rstd = 1/sqrt(var + eps), fp32 [rows], from the fixed-order C fold."""
    n = np.ascontiguousarray(part_n, dtype=np.float32)
    mu = np.ascontiguousarray(part_mu, dtype=np.float32)
    m2 = np.ascontiguousarray(part_m2, dtype=np.float32)
    rows, S = n.shape
    assert mu.shape == (rows, S) and m2.shape == (rows, S)
    mean = np.empty((rows,), np.float32)
    var = np.empty((rows,), np.float32)
    rstd = np.empty((rows,), np.float32)
    rc = load().fa_oracle_welford_combine_f32(_fptr(n), _fptr(mu), _fptr(m2), rows, S,
                                              ctypes.c_float(eps), _fptr(mean), _fptr(var),
                                              _fptr(rstd))
    if rc != 0:
        raise ValueError("fa_oracle_welford_combine_f32: bad sizes")
    return mean, var, rstd
