"""ctypes binding of libred.so: argument marshalling only."""
from __future__ import annotations

import ctypes
import os

import torch

RED_SUM, RED_MAX, RED_MIN, RED_PROD = 0, 1, 2, 3
RED_F32, RED_I32, RED_F16, RED_BF16, RED_I16, RED_U16, RED_U32 = 0, 1, 2, 3, 4, 5, 6
RED_OK, RED_EINVAL, RED_ECUDA, RED_ENOMEM = 0, -1, -2, -3
RED_MODE_AUTO, RED_MODE_TWO_PASS, RED_MODE_LAST_BLOCK, RED_MODE_ATOMIC = 0, 1, 2, 3
RED_KNOB_ROWS_GROUP, RED_KNOB_RAGGED_GROUP, RED_KNOB_COLPROD_SPLITS, RED_KNOB_FULL_CTAS_PER_SM = 1, 2, 3, 4
RED_KNOB_RAGGED_STAGED = 5
RED_KNOB_ROWS_ALIGNED = 6
RED_KNOB_COLS_LANES = 7

_OPS = {"sum": RED_SUM, "max": RED_MAX, "min": RED_MIN, "prod": RED_PROD}
# element type names of the column reductions and their sizes in bytes
_COL_DTYPES = {"f32": (RED_F32, 4), "i32": (RED_I32, 4), "f16": (RED_F16, 2), "bf16": (RED_BF16, 2),
               "i16": (RED_I16, 2), "u16": (RED_U16, 2), "u32": (RED_U32, 4)}
_TORCH_COL = {torch.float32: "f32", torch.int32: "i32", torch.float16: "f16", torch.bfloat16: "bf16",
              torch.int16: "i16"}
for _name, _key in (("uint16", "u16"), ("uint32", "u32")):
    if hasattr(torch, _name):
        _TORCH_COL[getattr(torch, _name)] = _key
_HERE = os.path.dirname(os.path.abspath(__file__))
_LIB_PATH = os.path.join(_HERE, "libred.so")
_lib = None

_i64, _int, _vp = ctypes.c_int64, ctypes.c_int, ctypes.c_void_p
_SIGNATURES = {
    "red_full": ([_int, _vp, _i64, _vp, _vp], _int),
    "red_full_noalloc": ([_int, _vp, _i64, _vp, _vp], _int),
    "red_full_stats": ([_vp, _i64, _vp, _vp], _int),
    "red_rows_stats": ([_vp, _i64, _i64, _vp, _vp], _int),
    "red_rows": ([_int, _vp, _i64, _i64, _int, _vp, _vp], _int),
    "red_rows_ragged": ([_int, _vp, _vp, _i64, _i64, _int, _vp, _vp], _int),
    "red_rows_thread": ([_int, _vp, _i64, _int, _int, _vp, _vp], _int),
    "red_colprod": ([_int, _vp, _i64, _i64, _vp, _vp], _int),
    "red_cols": ([_int, _int, _vp, _i64, _i64, _vp, _vp], _int),
    "red_cols_ld": ([_int, _int, _vp, _i64, _i64, _i64, _vp, _vp], _int),
    "red_full_typed": ([_int, _int, _vp, _i64, _vp, _vp], _int),
    "red_rows_typed": ([_int, _int, _vp, _i64, _i64, _int, _vp, _vp], _int),
    "red_set_full_mode": ([_int], _int),
    "red_get_full_mode": ([], _int),
    "red_set_knob": ([_int, _int], _int),
    "red_get_knob": ([_int], _int),
    "red_last_error": ([], ctypes.c_char_p),
    "red_release_workspace": ([], _int),
    "red_launch_count": ([], ctypes.c_uint64),
    "red_version": ([], _int),
}


class RedError(RuntimeError):
    """A libred call returned a non-OK status."""

    def __init__(self, status, message):
        super().__init__(f"libred status {status}: {message}")
        self.status = status


def lib_path() -> str:
    return _LIB_PATH


def lib():
    """The loaded libred.so (ctypes.CDLL).  Raises if it has not been built."""
    global _lib
    if _lib is None:
        if not os.path.exists(_LIB_PATH):
            raise RuntimeError(
                f"{_LIB_PATH} is missing: build it with int_tensor_reductions_gb300._build.build_lib() "
                "(or __graft_entry__.build()); there is no fallback implementation")
        l = ctypes.CDLL(_LIB_PATH)
        for name, (args, res) in _SIGNATURES.items():
            fn = getattr(l, name)
            fn.argtypes = args
            fn.restype = res
        _lib = l
    return _lib


def red_last_error() -> str:
    return lib().red_last_error().decode()


def _check(status):
    if status != RED_OK:
        raise RedError(status, red_last_error())


def _op(op) -> int:
    if isinstance(op, str):
        return _OPS[op]
    return int(op)


def _stream(stream, device) -> int:
    if stream is None:
        stream = torch.cuda.current_stream(device)
    return stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream)


def _need(t: torch.Tensor, name: str, dtypes, like: torch.Tensor | None = None, min_numel: int = 0):
    """t is a contiguous CUDA tensor of one of ``dtypes`` (None: any), on
    ``like``'s device when given, with at least ``min_numel`` elements."""
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if like is not None and t.device != like.device:
        raise ValueError(f"{name} is on {t.device}, x on {like.device}")
    if t.numel() < min_numel:
        raise ValueError(f"{name} must hold at least {min_numel} element(s)")
    if dtypes is None:
        if not t.is_contiguous():
            raise ValueError(f"{name} must be contiguous")
        return
    if t.dtype not in dtypes:
        raise ValueError(f"{name} must have dtype {dtypes}, got {t.dtype}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")


def red_full(op, x: torch.Tensor, out: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    """Reduce all of fp32 ``x`` to ``out`` (shape (1,)) on ``stream``."""
    _need(x, "x", (torch.float32,))
    if out is None:
        out = torch.empty(1, dtype=torch.float32, device=x.device)
    _need(out, "out", (torch.float32,), x, 1)
    with torch.cuda.device(x.device):
        _check(lib().red_full(_op(op), x.data_ptr(), x.numel(), out.data_ptr(), _stream(stream, x.device)))
    return out


def red_full_stats(x: torch.Tensor, out: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    """Sum, max, min and sum |x| of fp32 ``x`` from one read, into ``out`` (shape (4,))."""
    _need(x, "x", (torch.float32,))
    if out is None:
        out = torch.empty(4, dtype=torch.float32, device=x.device)
    _need(out, "out", (torch.float32,), x, 4)
    with torch.cuda.device(x.device):
        _check(lib().red_full_stats(x.data_ptr(), x.numel(), out.data_ptr(), _stream(stream, x.device)))
    return out


def red_rows_stats(x: torch.Tensor, out: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    """Per-row (sum, max, min, sum|x|) of a (rows, len) fp32 matrix from one read,
    into ``out`` of shape (rows, 4)."""
    _need(x, "x", (torch.float32,))
    if x.dim() != 2:
        raise ValueError("x must be 2-D (rows, len)")
    rows, length = x.shape
    if out is None:
        out = torch.empty((rows, 4), dtype=torch.float32, device=x.device)
    _need(out, "out", (torch.float32,), x)
    if out.numel() != 4 * rows:
        raise ValueError("out must hold 4 floats per row")
    with torch.cuda.device(x.device):
        _check(lib().red_rows_stats(x.data_ptr(), rows, length, out.data_ptr(), _stream(stream, x.device)))
    return out


def red_full_noalloc(op, x: torch.Tensor, out: torch.Tensor, stream=None) -> torch.Tensor:
    """red_full without any device allocation by the library: its scratch is a
    fixed array in the library (for callers that cannot let a library call
    cudaMalloc).  ``out`` must be given, so this wrapper allocates nothing
    either."""
    _need(x, "x", (torch.float32,))
    _need(out, "out", (torch.float32,), x, 1)
    with torch.cuda.device(x.device):
        _check(lib().red_full_noalloc(_op(op), x.data_ptr(), x.numel(), out.data_ptr(),
                                      _stream(stream, x.device)))
    return out


def red_rows(op, x: torch.Tensor, accum: bool = False, out: torch.Tensor | None = None,
             stream=None) -> torch.Tensor:
    """Per-row reduction of a (rows, len) row-major fp32 matrix into ``out[rows]``."""
    _need(x, "x", (torch.float32,))
    if x.dim() != 2:
        raise ValueError("x must be 2-D (rows, len)")
    rows, length = x.shape
    if out is None:
        if accum:
            raise ValueError("accum needs an existing out")
        out = torch.empty(rows, dtype=torch.float32, device=x.device)
    _need(out, "out", (torch.float32,), x)
    if out.numel() != rows:
        raise ValueError("out must have one element per row")
    with torch.cuda.device(x.device):
        _check(lib().red_rows(_op(op), x.data_ptr(), rows, length, int(bool(accum)), out.data_ptr(),
                              _stream(stream, x.device)))
    return out


def red_rows_thread(op, x: torch.Tensor, accum: bool = False, out: torch.Tensor | None = None,
                    stream=None) -> torch.Tensor:
    """Per-row reduction of a (rows, len) fp32 matrix, len <= 64, one thread per
    row with the page's thread-scope fold (fixed rounding order)."""
    _need(x, "x", (torch.float32,))
    if x.dim() != 2:
        raise ValueError("x must be 2-D (rows, len)")
    rows, length = x.shape
    if out is None:
        if accum:
            raise ValueError("accum needs an existing out")
        out = torch.empty(rows, dtype=torch.float32, device=x.device)
    _need(out, "out", (torch.float32,), x)
    if out.numel() != rows:
        raise ValueError("out must have one element per row")
    with torch.cuda.device(x.device):
        _check(lib().red_rows_thread(_op(op), x.data_ptr(), rows, length, int(bool(accum)), out.data_ptr(),
                                     _stream(stream, x.device)))
    return out


def red_rows_ragged(op, x: torch.Tensor, offsets: torch.Tensor, accum: bool = False,
                    out: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    """Per-row reduction of packed rows x[offsets[r]:offsets[r+1]]."""
    _need(x, "x", (torch.float32,))
    _need(offsets, "offsets", (torch.int64,), x, 1)
    rows = offsets.numel() - 1
    if rows < 0:
        raise ValueError("offsets needs rows + 1 entries")
    if out is None:
        if accum:
            raise ValueError("accum needs an existing out")
        out = torch.empty(rows, dtype=torch.float32, device=x.device)
    _need(out, "out", (torch.float32,), x)
    if out.numel() != rows:
        raise ValueError("out must have one element per row")
    with torch.cuda.device(x.device):
        _check(lib().red_rows_ragged(_op(op), x.data_ptr(), offsets.data_ptr(), rows, x.numel(),
                                     int(bool(accum)), out.data_ptr(), _stream(stream, x.device)))
    return out


def _col_dtype(x: torch.Tensor, dtype):
    key = dtype if dtype is not None else _TORCH_COL.get(x.dtype)
    if key not in _COL_DTYPES:
        raise ValueError(f"unsupported element type {x.dtype if dtype is None else dtype}")
    code, size = _COL_DTYPES[key]
    if x.element_size() != size:
        raise ValueError(f"element type {key} needs {size}-byte elements, x has {x.element_size()}")
    return code


def _row_strided(x: torch.Tensor, name: str = "x") -> int:
    """Row stride (elements) of a 2-D CUDA view whose rows are contiguous."""
    if not x.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if x.dim() != 2:
        raise ValueError(f"{name} must be 2-D (R, C)")
    R, C = x.shape
    if R > 1 and C > 1 and x.stride(1) != 1:
        raise ValueError(f"{name}'s rows must be contiguous (stride 1 along columns)")
    ld = x.stride(0) if R > 1 else C
    if ld < C:
        raise ValueError(f"{name}'s row stride {ld} is smaller than its {C} columns")
    return ld


def red_cols(op, x: torch.Tensor, out: torch.Tensor | None = None, stream=None, dtype=None) -> torch.Tensor:
    """Column reduction out[j] = op_i x[i, j] (op "sum", "max", "min" or
    "prod") of a (R, C) matrix of float32, int32, float16, bfloat16, int16,
    uint16 or uint32; ``dtype`` ("u16", "u32", ...) reads x's storage as that
    element type (same element size), e.g. int16 storage as uint16.  x may be
    a view with contiguous rows and a larger row stride (e.g. ``big[:, :C]``):
    the valid region of a wider tile."""
    ld = _row_strided(x)
    code = _col_dtype(x, dtype)
    R, C = x.shape
    if out is None:
        out = torch.empty(C, dtype=x.dtype, device=x.device)
    _need(out, "out", None, x)
    if out.element_size() != x.element_size():
        raise ValueError("out must have x's element size")
    if out.numel() != C:
        raise ValueError("out must have C elements")
    with torch.cuda.device(x.device):
        _check(lib().red_cols_ld(_op(op), code, x.data_ptr(), R, C, ld, out.data_ptr(), _stream(stream, x.device)))
    return out


def red_full_typed(op, x: torch.Tensor, out: torch.Tensor | None = None, stream=None, dtype=None) -> torch.Tensor:
    """op ("sum", "max", "min", "prod") over all of x, for every element type
    red_cols accepts; ``out`` (shape (1,)) has x's element type."""
    if not x.is_cuda or not x.is_contiguous():
        raise ValueError("x must be a contiguous CUDA tensor")
    code = _col_dtype(x, dtype)
    if out is None:
        out = torch.empty(1, dtype=x.dtype, device=x.device)
    _need(out, "out", None, x, 1)
    if out.element_size() != x.element_size():
        raise ValueError("out must have x's element size")
    with torch.cuda.device(x.device):
        _check(lib().red_full_typed(_op(op), code, x.data_ptr(), x.numel(), out.data_ptr(),
                                    _stream(stream, x.device)))
    return out


def red_rows_typed(op, x: torch.Tensor, accum: bool = False, out: torch.Tensor | None = None, stream=None,
                   dtype=None) -> torch.Tensor:
    """Per-row op of a (rows, len) matrix of any element type red_cols accepts,
    optionally folding the old out[r] in (accum)."""
    if not x.is_cuda or not x.is_contiguous():
        raise ValueError("x must be a contiguous CUDA tensor")
    if x.dim() != 2:
        raise ValueError("x must be 2-D (rows, len)")
    code = _col_dtype(x, dtype)
    rows, length = x.shape
    if out is None:
        if accum:
            raise ValueError("accum needs an existing out")
        out = torch.empty(rows, dtype=x.dtype, device=x.device)
    _need(out, "out", None, x)
    if out.element_size() != x.element_size():
        raise ValueError("out must have x's element size")
    if out.numel() != rows:
        raise ValueError("out must have one element per row")
    with torch.cuda.device(x.device):
        _check(lib().red_rows_typed(_op(op), code, x.data_ptr(), rows, length, int(bool(accum)), out.data_ptr(),
                                    _stream(stream, x.device)))
    return out


def red_colprod(x: torch.Tensor, out: torch.Tensor | None = None, stream=None, dtype=None) -> torch.Tensor:
    """TCOLPROD: out[j] = prod_i x[i, j] for a (R, C) matrix of any element
    type red_cols accepts (float32 rounds per step, integers wrap); x may have
    a row stride larger than C (the valid region of a wider tile)."""
    ld = _row_strided(x)
    code = _col_dtype(x, dtype)
    R, C = x.shape
    if out is None:
        out = torch.empty(C, dtype=x.dtype, device=x.device)
    _need(out, "out", None, x)
    if out.element_size() != x.element_size():
        raise ValueError("out must have x's element size")
    if out.numel() != C:
        raise ValueError("out must have C elements")
    with torch.cuda.device(x.device):
        _check(lib().red_cols_ld(RED_PROD, code, x.data_ptr(), R, C, ld, out.data_ptr(), _stream(stream, x.device)))
    return out


def red_set_full_mode(mode: int) -> None:
    _check(lib().red_set_full_mode(int(mode)))


def red_get_full_mode() -> int:
    return lib().red_get_full_mode()


def red_set_knob(k: int, value: int) -> None:
    _check(lib().red_set_knob(int(k), int(value)))


def red_get_knob(k: int) -> int:
    v = lib().red_get_knob(int(k))
    if v < 0:
        raise RedError(v, red_last_error())
    return v


def red_release_workspace() -> None:
    _check(lib().red_release_workspace())


def red_launch_count() -> int:
    return int(lib().red_launch_count())


def red_version() -> int:
    return lib().red_version()
