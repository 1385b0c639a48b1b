"""GB300-native fp32 / int32 axis reductions.

Python binding of libred.so (C ABI in ``include/red.h``): the functions below
carry the C entry points' names and only marshal arguments (torch tensors to
device pointers, sizes and the current CUDA stream); every step of every
reduction runs in the library's CUDA kernels.  There is no CPU fallback: if
libred.so is missing or CUDA is unavailable, the calls raise.

    red_full(op, x, out=None)                      op in "sum", "max", "min"
    red_rows(op, x, accum=False, out=None)         x: (rows, len) fp32
    red_rows_ragged(op, x, offsets, accum=False, out=None)
    red_colprod(x, out=None)                       x: (R, C) of any column element type
    red_cols(op, x, out=None)                      column sum / max / min / prod (x may be a
                                                   row-strided view: the C call red_cols_ld)
    red_full_typed / red_rows_typed                 full / per-row ops for every element type
    red_full_stats(x, out=None)                    sum, max, min, sum|x| in one read
    red_rows_stats(x, out=None)                    the same per row, out: (rows, 4)
    red_rows_thread(op, x, accum=False, out=None)  one thread per row, the page's fold order
    red_full_noalloc(op, x, out)                   red_full without any device allocation

Every call takes an optional ``stream`` (default: the current stream of x's
device) and returns ``out``.  Calls on one device must be ordered (one
stream, or streams ordered by events): they share the library's workspace.
"""
from ._binding import (  # noqa: F401
    RED_BF16, RED_EINVAL, RED_ECUDA, RED_ENOMEM, RED_F16, RED_F32, RED_I16, RED_I32, RED_KNOB_COLPROD_SPLITS,
    RED_KNOB_FULL_CTAS_PER_SM, RED_KNOB_RAGGED_GROUP, RED_KNOB_RAGGED_STAGED, RED_KNOB_ROWS_ALIGNED, RED_KNOB_ROWS_GROUP,
    RED_KNOB_COLS_LANES, RED_MAX, RED_MIN,
    RED_MODE_ATOMIC, RED_MODE_AUTO, RED_MODE_LAST_BLOCK, RED_MODE_TWO_PASS, RED_OK, RED_PROD, RED_SUM, RED_U16, RED_U32,
    RedError, lib, lib_path, red_colprod, red_cols, red_full, red_full_noalloc, red_full_stats, red_full_typed, red_get_full_mode, red_get_knob, red_last_error, red_launch_count,
    red_release_workspace, red_rows, red_rows_ragged, red_rows_stats, red_rows_thread, red_rows_typed, red_set_full_mode, red_set_knob, red_version,
)
