"""red_full_typed and red_rows_typed (sum / max / min / product of every
element type, rows with accum) on the GPU against the oracle, with the
tolerances of the column reductions: integer results and max / min bit for
bit; fp32 sums 1e-5 * sum|x|, fp32 products 5e-4 relative; half and
bfloat16 one unit in the last place plus the fp32 accumulation bound."""
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


def _decode(t, dtype):
    if dtype in ("f32", "f16"):
        return to_host(t).astype(np.float64)
    if dtype == "bf16":
        return t.to(torch.float64).cpu().numpy()
    return to_host(t).view(NP_INT[dtype]).astype(np.int64)


def _raw(t):
    return t.cpu().view(torch.int16 if t.element_size() == 2 else torch.int32).numpy()


def _ulp(v, mant):
    a = np.abs(v)
    # spacing of the type at |v|, floored at its subnormal spacing (a result
    # below the type's range rounds to a subnormal or zero)
    e = np.maximum(np.floor(np.log2(np.where(a > 0, a, 1.0))), EMIN[mant])
    return np.exp2(e - mant)


def _compare(got, op, dtype, ref, what, n):
    if dtype in NP_INT:
        bad = np.nonzero(got != ref)[0]
        assert bad.size == 0, f"{what}: {bad.size} mismatches, first {bad[0]}: {got[bad[0]]} vs {ref[bad[0]]}"
        return
    ref, ab = ref
    if op in ("max", "min"):
        bound = np.zeros_like(ref)
    elif dtype == "f32":
        bound = 1e-5 * ab if op == "sum" else 5e-4 * np.abs(ref)
    elif op == "sum":
        bound = _ulp(ref, MANT[dtype]) + 1e-5 * ab
    else:
        bound = _ulp(ref, MANT[dtype]) + n * 2.0**-24 * np.abs(ref)
    bad = np.nonzero(~(np.abs(got - ref) <= bound))[0]
    assert bad.size == 0, f"{what}: first bad {bad[0]}: got {got[bad[0]]!r} ref {ref[bad[0]]!r}"


@pytest.mark.parametrize("dtype", DTYPES)
@pytest.mark.parametrize("op", OPS)
def test_full(op, dtype):
    for n in (1, 7, 33, 1000, 65537, 1_000_003):
        x = synth.col_input(op, dtype, (n + 1,), n % 97, device="cuda")[1:]
        got = _decode(itr.red_full_typed(op, x, dtype=dtype), dtype)
        _compare(got, op, dtype, oracle.rows_typed(op, dtype, _raw(x), 1, n), f"{op} {dtype} n={n}", n)


@pytest.mark.parametrize("dtype", DTYPES)
@pytest.mark.parametrize("op", OPS)
def test_rows_with_accum(op, dtype):
    for rows, length in ((1, 1), (5, 3), (100, 17), (33, 64), (7, 1000), (3, 5000)):
        x = synth.col_input(op, dtype, (rows * length + 1,), rows + length, device="cuda")[1:].view(rows, length)
        old = synth.col_input(op, dtype, (rows,), 9, device="cuda")
        for accum in (False, True):
            out = old.clone()
            itr.red_rows_typed(op, x, accum=accum, out=out, dtype=dtype)
            ref = oracle.rows_typed(op, dtype, _raw(x), rows, length, accum, _raw(old))
            _compare(_decode(out, dtype), op, dtype, ref, f"{op} {dtype} {rows}x{length} accum={accum}", length + 1)


def test_empty_inputs():
    out = torch.full((1,), 9, dtype=torch.int32, device="cuda")
    itr.red_full_typed("prod", torch.empty(0, dtype=torch.int32, device="cuda"), out)
    assert int(out[0]) == 1
    itr.red_full_typed("sum", torch.empty(0, dtype=torch.int32, device="cuda"), out)
    assert int(out[0]) == 0
    with pytest.raises(itr.RedError):
        itr.red_full_typed("max", torch.empty(0, dtype=torch.int16, device="cuda"), torch.empty(1, dtype=torch.int16,
                                                                                               device="cuda"))
    o = torch.full((4,), 5, dtype=torch.int16, device="cuda")
    itr.red_rows_typed("sum", torch.empty((4, 0), dtype=torch.int16, device="cuda"), accum=True, out=o)
    assert o.cpu().tolist() == [5, 5, 5, 5]
    itr.red_rows_typed("prod", torch.empty((4, 0), dtype=torch.int16, device="cuda"), out=o)
    assert o.cpu().tolist() == [1, 1, 1, 1]


def test_int32_sum_wraps():
    """2^31 - 1 + 1 wraps to -2^31 in int32 (bit for bit with the oracle)."""
    x = torch.tensor([2**31 - 1, 1], dtype=torch.int32, device="cuda")
    assert int(itr.red_full_typed("sum", x)[0]) == -2**31


@pytest.mark.parametrize("dtype", DTYPES)
@pytest.mark.parametrize("op", OPS)
def test_rows_of_a_block_or_less(op, dtype):
    """Rows of 2 to 32 bytes (one 32-byte block holds 1 to 16 of them) and of
    2 to 32 whole blocks, from a 32-byte aligned base, row counts that leave
    a partial block or a partial warp of blocks, results
    written as vectors (aligned out) and element by element (out one element
    off its alignment), with and without accum; the element just outside out
    keeps its value."""
    size = 2 if dtype in ("f16", "bf16", "i16", "u16") else 4
    for length in (1, 2, 4, 8, 16, 32, 64, 128, 256, 512):
        if length * size > 1024:
            continue
        for rows in ((1, 15, 17, 1000, 100_003) if length * size <= 32 else (1, 3, 33, 1000, 20_003)):
            x = synth.col_input(op, dtype, (rows, length), rows + length, device="cuda")
            assert x.data_ptr() % 32 == 0
            old_full = synth.col_input(op, dtype, (rows + 1,), length, device="cuda")
            for shift in (0, 1):
                old = old_full[shift:shift + rows]
                for accum in (False, True):
                    buf = old_full.clone()  # the element outside out must not change
                    out = buf[shift:shift + rows]
                    itr.red_rows_typed(op, x, accum=accum, out=out, dtype=dtype)
                    ref = oracle.rows_typed(op, dtype, _raw(x), rows, length, accum, _raw(old))
                    what = f"{op} {dtype} {rows}x{length} shift={shift} accum={accum}"
                    _compare(_decode(out, dtype), op, dtype, ref, what, length + 1)
                    edge = 0 if shift else rows
                    assert _raw(buf[edge:edge + 1]).tolist() == _raw(old_full[edge:edge + 1]).tolist(), what
