"""red_cols (column sum / max / min / product, TCOLPROD and its siblings)
for every element type of the pages' A2A3 / A5 lists, against the oracle:
integer results and max / min bit for bit; fp32 sums within 1e-5 * sum|x|
and fp32 products within 5e-4 relative (the workload's tolerances); half and
bfloat16 within one unit in the last place of the result type plus the fp32
accumulation bound (R * 2^-24 relative for products, 1e-5 * sum|x| for sums)
-- the result is one rounding of an fp32 accumulation.  Shapes cover the
256-bit, 128-bit and scalar column paths (row length and base alignment),
row splits and the workload sizes."""
import math

import numpy as np
import pytest
import torch

import oracle
import int_tensor_reductions_gb300 as itr
from int_tensor_reductions_gb300 import synth
from gpu_util import lib_ready, to_host

pytestmark = pytest.mark.gpu

DTYPES = ["f32", "i32", "u32", "f16", "bf16", "i16", "u16"]
OPS = ["sum", "max", "min", "prod"]
NP_INT = {"i32": np.int32, "u32": np.uint32, "i16": np.int16, "u16": np.uint16}
MANT = {"f16": 10, "bf16": 7}
EMIN = {10: -14, 7: -126}  # smallest normal exponent of half / bfloat16


@pytest.fixture(scope="module", autouse=True)
def _lib():
    lib_ready()
    yield
    itr.red_set_knob(itr.RED_KNOB_COLPROD_SPLITS, 0)
    itr.red_set_knob(itr.RED_KNOB_COLS_LANES, 0)


def _decode(t: torch.Tensor, dtype: str) -> np.ndarray:
    """GPU result -> float64 (floating types) or int64 (integer types)."""
    if dtype == "f32":
        return to_host(t).astype(np.float64)
    if dtype == "f16":
        return to_host(t).astype(np.float64)
    if dtype == "bf16":
        return t.to(torch.float64).cpu().numpy()
    return to_host(t).view(NP_INT[dtype]).astype(np.int64)


def _ulp(v, mant):
    a = np.abs(v)
    # spacing of the type at |v|, floored at its subnormal spacing (a result
    # below the type's range rounds to a subnormal or zero)
    e = np.maximum(np.floor(np.log2(np.where(a > 0, a, 1.0))), EMIN[mant])
    return np.exp2(e - mant)


def check_cols(op, dtype, x: torch.Tensor, what, cols=None):
    R, C = x.shape
    out = itr.red_cols(op, x, dtype=dtype)
    got = _decode(out, dtype)
    xh = x.cpu().contiguous()  # x may be a row-strided view
    if cols is not None:
        xh = xh[:, cols].contiguous()
        got = got[cols]
    raw = xh.view(torch.int16 if xh.element_size() == 2 else torch.int32).numpy()
    ncol = xh.shape[1]
    if dtype in NP_INT:
        ref = oracle.cols(op, dtype, raw, R, ncol)
        bad = np.nonzero(got != ref)[0]
        assert bad.size == 0, f"{what}: {bad.size} mismatches, first col {bad[0]}: {got[bad[0]]} vs {ref[bad[0]]}"
        return
    ref, ab = oracle.cols(op, dtype, raw, R, ncol)
    if op in ("max", "min"):
        bound = np.zeros_like(ref)
    elif dtype == "f32":
        bound = 1e-5 * ab if op == "sum" else 5e-4 * np.abs(ref)
    elif op == "sum":
        bound = _ulp(ref, MANT[dtype]) + 1e-5 * ab
    else:
        bound = _ulp(ref, MANT[dtype]) + R * 2.0**-24 * np.abs(ref)
    err = np.abs(got - ref)
    bad = np.nonzero(~(err <= bound))[0]
    assert bad.size == 0, (f"{what}: {bad.size} out of tolerance, first col {bad[0]}: got {got[bad[0]]!r} "
                           f"ref {ref[bad[0]]!r} bound {bound[bad[0]]!r}")


@pytest.mark.parametrize("dtype", DTYPES)
@pytest.mark.parametrize("op", OPS)
def test_shapes_and_paths(op, dtype):
    for R, C in [(1, 1), (3, 5), (37, 129), (100, 1000), (64, 16), (5, 8), (129, 257), (1000, 96), (33, 4100)]:
        x = synth.col_input(op, dtype, (R * C + 1,), R * 7 + C, device="cuda")
        check_cols(op, dtype, x[:R * C].view(R, C), f"{op} {dtype} {R}x{C}")
        check_cols(op, dtype, x[1:].view(R, C), f"{op} {dtype} {R}x{C} base+1")


@pytest.mark.parametrize("dtype", DTYPES)
@pytest.mark.parametrize("splits", [1, 3, 64])
def test_forced_row_splits(dtype, splits):
    itr.red_set_knob(itr.RED_KNOB_COLPROD_SPLITS, splits)
    try:
        for op in OPS:
            x = synth.col_input(op, dtype, (700, 1040), splits, device="cuda")
            check_cols(op, dtype, x, f"{op} {dtype} splits={splits}")
    finally:
        itr.red_set_knob(itr.RED_KNOB_COLPROD_SPLITS, 0)


@pytest.mark.parametrize("dtype", ["f32", "i32", "f16", "u16"])
@pytest.mark.parametrize("R,C", [(5000, 256), (2000, 8192), (777, 33000), (65, 40000), (3, 70000)])
def test_tall_wide_and_ragged_tiles(R, C, dtype):
    """One column tile of 5000 rows, 32 tiles of 2000 rows, 129 tiles with a
    ragged last one, and very wide matrices of few rows (many tiles, few or
    no row splits)."""
    for op in ("prod", "sum", "max"):
        x = synth.col_input(op, dtype, (R, C), R + C, device="cuda")
        check_cols(op, dtype, x, f"{op} {dtype} {R}x{C}")


@pytest.mark.parametrize("lanes", [1, 2, 4, 8, 16, 32])
def test_every_lanes_per_row_setting(lanes):
    """Column tiles of 1 to 32 lanes per row (the automatic choice takes 8
    for matrices of many rows, 32 for short ones), with the automatic and a
    forced split count."""
    itr.red_set_knob(itr.RED_KNOB_COLS_LANES, lanes)
    try:
        for dtype in ("f32", "i32", "bf16", "u16"):
            for op, (R, C) in (("prod", (300, 1032)), ("sum", (2000, 520)), ("max", (64, 4104)), ("min", (3, 136))):
                x = synth.col_input(op, dtype, (R, C), R + lanes, device="cuda")
                check_cols(op, dtype, x, f"{op} {dtype} {R}x{C} lanes={lanes}")
                itr.red_set_knob(itr.RED_KNOB_COLPROD_SPLITS, 5)
                try:
                    check_cols(op, dtype, x, f"{op} {dtype} {R}x{C} lanes={lanes} splits=5")
                finally:
                    itr.red_set_knob(itr.RED_KNOB_COLPROD_SPLITS, 0)
    finally:
        itr.red_set_knob(itr.RED_KNOB_COLS_LANES, 0)


def test_int_wrap_closed_forms():
    for c, R, dtype, ref in [(2, 15, "i16", -32768), (2, 16, "i16", 0), (3, 11, "i16", 177147 - 3 * 65536),
                             (3, 11, "u16", 177147 % 65536), (2, 32, "u32", 0), (3, 21, "u32", 3**21 % 2**32),
                             (2, 31, "i32", -2**31)]:
        x = torch.full((R, 48), c, dtype=synth.COL_STORAGE[dtype], device="cuda")
        got = _decode(itr.red_colprod(x, dtype=dtype), dtype)
        assert (got == ref).all(), (c, R, dtype)


def test_half_sum_rounds_once():
    """2048 rows of half 1.0 + 2^-10: the fp32 column sum is exact (2048 +
    2) and rounds once to half (2050, representable); rounding each partial
    sum to half instead would stall at 2048."""
    x = torch.full((2048, 64), 1.0 + 2.0**-10, dtype=torch.float16, device="cuda")
    assert (to_host(itr.red_cols("sum", x)).astype(np.float64) == 2050.0).all()


@pytest.mark.parametrize("dtype", ["f16", "bf16"])
def test_workload_size_16bit(dtype):
    """4096 x 16384 of a 16-bit float type (sampled columns)."""
    for op in ("prod", "sum"):
        x = synth.col_input(op, dtype, (4096, 16384), 3, device="cuda")
        cols = np.unique(np.concatenate([np.random.default_rng(1).choice(16384, 512, replace=False), [0, 16383]]))
        check_cols(op, dtype, x, f"{op} {dtype} 4096x16384", cols=cols)


@pytest.mark.parametrize("dtype", ["i16", "u16", "u32"])
def test_workload_size_int(dtype):
    for op in ("prod", "sum", "max"):
        x = synth.col_input(op, dtype, (64, 65536), 4, device="cuda")
        check_cols(op, dtype, x, f"{op} {dtype} 64x65536")


def test_early_return_every_type():
    for dtype in DTYPES:
        st = synth.COL_STORAGE[dtype]
        out = torch.full((5,), 3, dtype=st, device="cuda")
        itr.red_cols("max", torch.empty((0, 5), dtype=st, device="cuda"), out, dtype=dtype)
        assert (out.cpu() == 3).all(), dtype


@pytest.mark.parametrize("dtype", DTYPES)
@pytest.mark.parametrize("R,C,ld", [(37, 100, 104), (500, 1040, 1056), (64, 4096, 5000), (3, 1, 9), (1, 17, 40)])
def test_valid_region_of_a_wider_matrix(R, C, ld, dtype):
    """TCOLPROD over the valid region R x C of a row-major matrix whose rows
    are ld elements apart (pto-isa docs, "TCOLPROD", "Math Interpretation":
    R = ValidRow, C = ValidCol).  The columns past C hold values that would
    change every result if they were read (NaN for floats; for integers the
    type's extreme values)."""
    for op in OPS:
        full = synth.col_input(op, dtype, (R, ld), R * 3 + C, device="cuda")
        pad = full[:, C:]
        if full.is_floating_point():
            pad.fill_(float("nan"))
        else:
            pad.fill_(-1 if dtype in ("u16", "u32") else torch.iinfo(full.dtype).min)
        check_cols(op, dtype, full[:, :C], f"{op} {dtype} {R}x{C} ld={ld}")
    p = itr.red_colprod(synth.col_input("prod", dtype, (R, ld), 5, device="cuda")[:, :C], dtype=dtype)
    assert p.numel() == C
