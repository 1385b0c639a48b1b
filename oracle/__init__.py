"""CPU oracle for the axis reductions -- TEST INFRASTRUCTURE ONLY.

Only the test suite, ``__graft_entry__.smoke()`` and ``bench.py``'s CPU-baseline
leg (and its ``--impl reference`` arm) may import this package.  The product
path (``int_tensor_reductions_gb300`` and its CUDA library) never does, and the
two share no code: this package wraps ``oracle.c``, a plain single-threaded C
restatement of what each reduction computes (see the header of ``oracle.c``
for the passages it follows), through ``ctypes`` on host numpy arrays.

The shared library is built with ``gcc -O2`` (no fast-math, no OpenMP) on first
use, or by :func:`build`.
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_LIB = os.path.join(_HERE, "liboracle.so")

_lib = None


def build(force: bool = False) -> str:
    """Compile ``oracle.c`` into ``liboracle.so`` beside it; return its path."""
    stale = (not os.path.exists(_LIB)) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC)
    if force or stale:
        tmp = _LIB + ".tmp%d" % os.getpid()
        subprocess.run(
            ["gcc", "-std=c99", "-O2", "-fno-fast-math", "-fPIC", "-shared",
             "-Wall", "-Wextra", "-o", tmp, _SRC, "-lm"],
            check=True,
        )
        os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    if _lib is not None:
        return _lib
    # ORACLE_LIB: a deliberately broken build of oracle.c, used only by the
    # test that checks the pins catch planted mistakes
    lib = ctypes.CDLL(os.environ.get("ORACLE_LIB") or build())
    i64, i32 = ctypes.c_int64, ctypes.c_int
    vp = ctypes.c_void_p
    sigs = {
        "orc_full_sum": [vp, i64, vp, vp],
        "orc_full_max": [vp, i64, vp],
        "orc_full_min": [vp, i64, vp],
        "orc_rows_sum": [vp, i64, i64, i32, vp, vp, vp],
        "orc_rows_max": [vp, i64, i64, i32, vp, vp],
        "orc_rows_min": [vp, i64, i64, i32, vp, vp],
        "orc_ragged_sum": [vp, vp, i64, i32, vp, vp, vp],
        "orc_ragged_max": [vp, vp, i64, i32, vp, vp],
        "orc_ragged_min": [vp, vp, i64, i32, vp, vp],
        "orc_colprod_f32": [vp, i64, i64, vp, vp],
        "orc_colprod_i32": [vp, i64, i64, vp],
    }
    lib.orc_thread_sum.argtypes = [vp, i64, i32, ctypes.c_float]
    lib.orc_thread_sum.restype = ctypes.c_float
    lib.orc_half_to_double.argtypes = [ctypes.c_uint16]
    lib.orc_half_to_double.restype = ctypes.c_double
    lib.orc_bf16_to_double.argtypes = [ctypes.c_uint16]
    lib.orc_bf16_to_double.restype = ctypes.c_double
    sigs["orc_cols_f"] = [i32, i32, vp, i64, i64, vp, vp]
    sigs["orc_cols_i"] = [i32, i32, vp, i64, i64, vp]
    sigs["orc_rows_typed_f"] = [i32, i32, vp, i64, i64, i32, vp, vp, vp]
    sigs["orc_rows_typed_i"] = [i32, i32, vp, i64, i64, i32, vp, vp]
    for name, args in sigs.items():
        fn = getattr(lib, name)
        fn.argtypes = args
        fn.restype = ctypes.c_int
    _lib = lib
    return lib


class OracleError(ValueError):
    """The oracle rejected its arguments (status -1)."""


def _ptr(a):
    return None if a is None else a.ctypes.data


def _f32(a):
    a = np.ascontiguousarray(a, dtype=np.float32)
    return a


def _check(status, what):
    if status != 0:
        raise OracleError(f"oracle rejected {what} (status {status})")


# --------------------------------------------------------------------- full

def full_sum(x):
    """Return (sum, sum|x|) of a 1-D fp32 vector, both as Python floats (double)."""
    x = _f32(x).reshape(-1)
    s = ctypes.c_double()
    a = ctypes.c_double()
    _check(_load().orc_full_sum(_ptr(x), x.size, ctypes.byref(s), ctypes.byref(a)), "full_sum")
    return s.value, a.value


def full_max(x):
    x = _f32(x).reshape(-1)
    o = np.zeros(1, np.float32)
    _check(_load().orc_full_max(_ptr(x), x.size, _ptr(o)), "full_max")
    return o[0]


def full_min(x):
    x = _f32(x).reshape(-1)
    o = np.zeros(1, np.float32)
    _check(_load().orc_full_min(_ptr(x), x.size, _ptr(o)), "full_min")
    return o[0]


def full(op, x):
    """op in {"sum","max","min"}; sum returns (sum, abs_sum), max/min a float32."""
    return {"sum": full_sum, "max": full_max, "min": full_min}[op](x)


# ---------------------------------------------------------------- dense rows

def rows(op, x, rows_, len_, accum=False, dst_old=None):
    """Per-row reduction of a row-major ``rows_ x len_`` fp32 matrix.

    sum -> (float64[rows], abs float64[rows]); max/min -> float32[rows].
    """
    x = _f32(x).reshape(-1)
    if x.size != rows_ * len_:
        raise OracleError("x has the wrong size")
    d = None if not accum else _f32(dst_old).reshape(-1)
    lib = _load()
    if op == "sum":
        out = np.zeros(rows_, np.float64)
        ab = np.zeros(rows_, np.float64)
        _check(lib.orc_rows_sum(_ptr(x), rows_, len_, int(accum), _ptr(d), _ptr(out), _ptr(ab)), "rows_sum")
        return out, ab
    out = np.zeros(rows_, np.float32)
    fn = {"max": lib.orc_rows_max, "min": lib.orc_rows_min}[op]
    _check(fn(_ptr(x), rows_, len_, int(accum), _ptr(d), _ptr(out)), "rows_" + op)
    return out


# --------------------------------------------------------------- ragged rows

def ragged(op, x, offsets, accum=False, dst_old=None):
    """Per-row reduction of packed rows x[offsets[r]:offsets[r+1]]."""
    x = _f32(x).reshape(-1)
    off = np.ascontiguousarray(offsets, dtype=np.int64).reshape(-1)
    nrows = off.size - 1
    if nrows < 0 or off[-1] > x.size:
        raise OracleError("bad offsets")
    d = None if not accum else _f32(dst_old).reshape(-1)
    lib = _load()
    if op == "sum":
        out = np.zeros(nrows, np.float64)
        ab = np.zeros(nrows, np.float64)
        _check(lib.orc_ragged_sum(_ptr(x), _ptr(off), nrows, int(accum), _ptr(d), _ptr(out), _ptr(ab)),
               "ragged_sum")
        return out, ab
    out = np.zeros(nrows, np.float32)
    fn = {"max": lib.orc_ragged_max, "min": lib.orc_ragged_min}[op]
    _check(fn(_ptr(x), _ptr(off), nrows, int(accum), _ptr(d), _ptr(out)), "ragged_" + op)
    return out


# ------------------------------------------------------------------ TCOLPROD

def colprod_f32(x, R, C, out_f=None, want_double=False):
    """Column products of a row-major R x C fp32 matrix.

    Returns the fp32 result (written into ``out_f`` if given, so that the
    early return for R == 0 or C == 0 leaves it untouched), and with
    ``want_double`` also the double-precision products.
    """
    x = _f32(x).reshape(-1)
    if x.size != R * C:
        raise OracleError("x has the wrong size")
    if out_f is None:
        out_f = np.zeros(C, np.float32)
    out_d = np.zeros(C, np.float64) if want_double else None
    _check(_load().orc_colprod_f32(_ptr(x), R, C, _ptr(out_f), _ptr(out_d)), "colprod_f32")
    return (out_f, out_d) if want_double else out_f


def thread_sum(a, accum=False, dst=0.0):
    """The sm100_packed thread-scope sum of a 1-D vector in the page's fp32
    rounding order (see orc_thread_sum in oracle.c); returns a float32."""
    a = _f32(a).reshape(-1)
    return np.float32(_load().orc_thread_sum(_ptr(a), a.size, int(bool(accum)), float(np.float32(dst))))


def thread_rows_sum(x, rows, len_, accum=False, dst_old=None):
    """thread_sum of every row of a row-major rows x len_ matrix (float32[rows])."""
    x = _f32(x).reshape(rows, len_)
    d = np.zeros(rows, np.float32) if dst_old is None else _f32(dst_old).reshape(-1)
    return np.array([thread_sum(x[r], accum, d[r]) for r in range(rows)], np.float32)


def colprod_i32(x, R, C, out=None):
    """Wrapping int32 column products of a row-major R x C int32 matrix."""
    x = np.ascontiguousarray(x, dtype=np.int32).reshape(-1)
    if x.size != R * C:
        raise OracleError("x has the wrong size")
    if out is None:
        out = np.zeros(C, np.int32)
    _check(_load().orc_colprod_i32(_ptr(x), R, C, _ptr(out)), "colprod_i32")
    return out


# ---------------------------------------------------- column reductions

COL_DTYPES = {"f32": 0, "i32": 1, "f16": 2, "bf16": 3, "i16": 4, "u16": 5, "u32": 6}
COL_OPS = {"sum": 0, "max": 1, "min": 2, "prod": 3}
_COL_BYTES = {"f32": 4, "i32": 4, "u32": 4, "f16": 2, "bf16": 2, "i16": 2, "u16": 2}


def half_to_double(bits: int) -> float:
    return _load().orc_half_to_double(int(bits) & 0xFFFF)


def bf16_to_double(bits: int) -> float:
    return _load().orc_bf16_to_double(int(bits) & 0xFFFF)


def cols(op, dtype, x, R, C, out=None):
    """Column reductions of a row-major R x C matrix given as raw element
    storage (any numpy array whose bytes are the R*C elements of ``dtype``).

    Floating types return (float64[C] result, float64[C] sum|x|); integer
    types return int64[C] (the result as the type, sign-extended).  With
    R == 0 or C == 0 the oracle returns early: ``out`` (if given) is left as
    it is and returned.
    """
    raw = np.ascontiguousarray(x).view(np.uint8).reshape(-1)
    if raw.size != R * C * _COL_BYTES[dtype]:
        raise OracleError("x has the wrong size")
    lib = _load()
    if dtype in ("f32", "f16", "bf16"):
        res = np.zeros(C, np.float64) if out is None else out
        ab = np.zeros(C, np.float64)
        _check(lib.orc_cols_f(COL_OPS[op], COL_DTYPES[dtype], _ptr(raw), R, C, _ptr(res), _ptr(ab)), "cols_f")
        return res, ab
    res = np.zeros(C, np.int64) if out is None else out
    _check(lib.orc_cols_i(COL_OPS[op], COL_DTYPES[dtype], _ptr(raw), R, C, _ptr(res)), "cols_i")
    return res


def rows_typed(op, dtype, x, rows_, len_, accum=False, dst_old=None):
    """Per-row op of a row-major rows_ x len_ matrix in raw element storage
    (a full vector is rows_ = 1).  Floating types return (float64[rows]
    result, float64[rows] sum|x|); integer types int64[rows]."""
    raw = np.ascontiguousarray(x).view(np.uint8).reshape(-1)
    if raw.size != rows_ * len_ * _COL_BYTES[dtype]:
        raise OracleError("x has the wrong size")
    d = None if not accum else np.ascontiguousarray(dst_old).view(np.uint8).reshape(-1)
    lib = _load()
    if dtype in ("f32", "f16", "bf16"):
        out = np.zeros(rows_, np.float64)
        ab = np.zeros(rows_, np.float64)
        _check(lib.orc_rows_typed_f(COL_OPS[op], COL_DTYPES[dtype], _ptr(raw), rows_, len_, int(bool(accum)),
                                    _ptr(d), _ptr(out), _ptr(ab)), "rows_typed_f")
        return out, ab
    out = np.zeros(rows_, np.int64)
    _check(lib.orc_rows_typed_i(COL_OPS[op], COL_DTYPES[dtype], _ptr(raw), rows_, len_, int(bool(accum)),
                                _ptr(d), _ptr(out)), "rows_typed_i")
    return out
