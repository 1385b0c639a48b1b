"""Seeded random cases of the entry points against the oracle: sizes,
base alignments, operators, element types, accum, row strides and every
mapping choice (grid stage, lanes per row, aligned or general row kernel,
ragged mapping, column row splits and lanes per column-tile row) drawn at
random, so that combinations the hand-picked shapes of the
other files do not name are covered too.  Same tolerances as those files:
integer and max / min results bit for bit, fp32 sums within 1e-5 * sum|x|,
fp32 products within 5e-4 relative, half and bfloat16 within one unit in
the last place plus the fp32 accumulation bound."""
import numpy as np
import pytest
import torch

import oracle
import int_tensor_reductions_gb300 as itr
from int_tensor_reductions_gb300 import synth
from gpu_util import check_exact, check_sum, lib_ready, to_host
from test_gpu_cols import check_cols
from test_gpu_typed import _compare, _decode, _raw

pytestmark = pytest.mark.gpu

OPS3 = ("sum", "max", "min")
DTYPES = ["f32", "i32", "u32", "f16", "bf16", "i16", "u16"]
N_CASES = 40


@pytest.fixture(scope="module", autouse=True)
def _lib():
    lib_ready()
    yield
    _reset()


def _reset():
    itr.red_set_full_mode(itr.RED_MODE_AUTO)
    for k in (itr.RED_KNOB_ROWS_GROUP, itr.RED_KNOB_RAGGED_GROUP, itr.RED_KNOB_COLPROD_SPLITS,
              itr.RED_KNOB_RAGGED_STAGED, itr.RED_KNOB_ROWS_ALIGNED, itr.RED_KNOB_COLS_LANES):
        itr.red_set_knob(k, 0)


def _shifted(x: torch.Tensor, n: int, shift: int) -> torch.Tensor:
    """n elements of x starting at element shift (x holds n + 8)."""
    return x[shift:shift + n]


@pytest.mark.parametrize("case", range(N_CASES))
def test_full(case):
    gen = np.random.default_rng(1000 + case)
    n = int(gen.choice([1, 7, 8, 9, 63, 1000, 65537, 300001, 2_000_003]))
    if gen.random() < 0.5:
        n = int(gen.integers(1, 400_000))
    shift = int(gen.integers(0, 8))
    mode = int(gen.integers(0, 4))
    x = _shifted(synth.uniform((n + 8,), -4.0, 4.0, case, device="cuda"), n, shift)
    xh = to_host(x)
    itr.red_set_full_mode(mode)
    try:
        for op in OPS3:
            got = to_host(itr.red_full(op, x))
            what = f"case {case}: n={n} shift={shift} mode={mode} {op}"
            if op == "sum":
                s, a = oracle.full_sum(xh)
                check_sum(got, [s], [a], what)
            else:
                check_exact(got, np.array([oracle.full(op, xh)], np.float32), what)
    finally:
        _reset()


@pytest.mark.parametrize("case", range(N_CASES))
def test_rows(case):
    gen = np.random.default_rng(2000 + case)
    length = int(gen.choice([1, 3, 8, 17, 64, 65, 100, 1023, 1024, 4097, 40000]))
    rows = int(gen.integers(1, max(2, min(3000, 2_000_000 // length))))
    shift = int(gen.integers(0, 8))
    g = int(gen.choice([0, 0, 1, 2, 4, 8, 16, 32]))
    accum = bool(gen.integers(0, 2))
    x = _shifted(synth.uniform((rows * length + 8,), -4.0, 4.0, case, device="cuda"), rows * length,
                 shift).view(rows, length)
    dst = synth.uniform((rows,), -1.0, 1.0, case + 1, device="cuda")
    xh, dh = to_host(x), to_host(dst)
    aligned = int(gen.choice([0, 2]))  # 2: the general row kernel even for rows of whole 32-byte blocks
    itr.red_set_knob(itr.RED_KNOB_ROWS_GROUP, g)
    itr.red_set_knob(itr.RED_KNOB_ROWS_ALIGNED, aligned)
    try:
        for op in OPS3:
            out = dst.clone()
            itr.red_rows(op, x, accum=accum, out=out)
            what = f"case {case}: {rows}x{length} shift={shift} G={g} aligned={aligned} accum={accum} {op}"
            if op == "sum":
                s, a = oracle.rows("sum", xh, rows, length, accum, dh)
                check_sum(to_host(out), s, a, what)
            else:
                check_exact(to_host(out), oracle.rows(op, xh, rows, length, accum, dh), what)
    finally:
        _reset()


@pytest.mark.parametrize("case", range(N_CASES))
def test_ragged(case):
    gen = np.random.default_rng(3000 + case)
    maxlen = int(gen.choice([1, 3, 6, 12, 40, 200, 3000]))
    rows = int(gen.integers(1, 6000))
    lens = gen.integers(0, maxlen + 1, size=rows)
    if gen.random() < 0.3:
        lens[int(gen.integers(0, rows))] = int(gen.choice([9000, 30000]))  # a row longer than a staged tile
    off = np.zeros(rows + 1, np.int64)
    off[1:] = np.cumsum(lens)
    nnz = int(off[-1])
    shift = int(gen.integers(0, 8))
    mode = int(gen.integers(0, 3))
    g = int(gen.choice([0, 0, 1, 2, 4, 32]))
    accum = bool(gen.integers(0, 2))
    x = _shifted(synth.uniform((nnz + 8,), -4.0, 4.0, case, device="cuda"), nnz, shift)
    offd = torch.from_numpy(off).cuda()
    dst = synth.uniform((rows,), -1.0, 1.0, case + 1, device="cuda")
    xh, dh = to_host(x), to_host(dst)
    itr.red_set_knob(itr.RED_KNOB_RAGGED_STAGED, mode)
    itr.red_set_knob(itr.RED_KNOB_RAGGED_GROUP, g)
    try:
        for op in OPS3:
            out = dst.clone()
            itr.red_rows_ragged(op, x, offd, accum=accum, out=out)
            what = f"case {case}: {rows} rows up to {maxlen} shift={shift} mode={mode} G={g} accum={accum} {op}"
            if op == "sum":
                s, a = oracle.ragged("sum", xh, off, accum, dh)
                check_sum(to_host(out), s, a, what)
            else:
                check_exact(to_host(out), oracle.ragged(op, xh, off, accum, dh), what)
    finally:
        _reset()


@pytest.mark.parametrize("case", range(N_CASES))
def test_cols(case):
    gen = np.random.default_rng(4000 + case)
    dtype = DTYPES[int(gen.integers(0, len(DTYPES)))]
    op = ("sum", "max", "min", "prod")[int(gen.integers(0, 4))]
    R = int(gen.choice([1, 2, 7, 64, 127, 128, 129, 500, 3000]))
    C = int(gen.choice([1, 5, 8, 16, 33, 64, 100, 256, 1000, 4096, 5000]))
    ld = C + int(gen.choice([0, 0, 1, 8, 16, 37]))
    shift = int(gen.integers(0, 4))
    splits = int(gen.choice([0, 0, 1, 2, 7, 64]))
    full = synth.col_input(op, dtype, (R * ld + shift,), case, device="cuda")
    x = full[shift:].view(R, ld)[:, :C]
    lanes = int(gen.choice([0, 0, 1, 2, 4, 8, 16, 32]))
    itr.red_set_knob(itr.RED_KNOB_COLPROD_SPLITS, splits)
    itr.red_set_knob(itr.RED_KNOB_COLS_LANES, lanes)
    try:
        check_cols(op, dtype, x,
                   f"case {case}: {op} {dtype} {R}x{C} ld={ld} shift={shift} splits={splits} lanes={lanes}")
    finally:
        _reset()


@pytest.mark.parametrize("case", range(N_CASES))
def test_typed_rows(case):
    gen = np.random.default_rng(5000 + case)
    dtype = DTYPES[int(gen.integers(0, len(DTYPES)))]
    op = ("sum", "max", "min", "prod")[int(gen.integers(0, 4))]
    length = int(gen.choice([1, 2, 3, 4, 8, 16, 17, 32, 64, 128, 100, 1000, 5000]))
    rows = int(gen.integers(1, max(2, min(4000, 1_000_000 // length))))
    shift = int(gen.integers(0, 2))
    accum = bool(gen.integers(0, 2))
    full = synth.col_input(op, dtype, (rows * length + 1,), case, device="cuda")
    x = full[shift:shift + rows * length].view(rows, length)
    old = synth.col_input(op, dtype, (rows,), case + 1, device="cuda")
    out = old.clone()
    itr.red_rows_typed(op, x, accum=accum, out=out, dtype=dtype)
    ref = oracle.rows_typed(op, dtype, _raw(x), rows, length, accum, _raw(old))
    _compare(_decode(out, dtype), op, dtype, ref,
             f"case {case}: {op} {dtype} {rows}x{length} shift={shift} accum={accum}", length + 1)


@pytest.mark.parametrize("case", range(N_CASES))
def test_thread_rows(case):
    gen = np.random.default_rng(6000 + case)
    length = int(gen.integers(1, 65))
    rows = int(gen.integers(1, 5000))
    shift = int(gen.integers(0, 8))
    accum = bool(gen.integers(0, 2))
    x = _shifted(synth.uniform((rows * length + 8,), -4.0, 4.0, case, device="cuda"), rows * length,
                 shift).view(rows, length)
    dst = synth.uniform((rows,), -1.0, 1.0, case + 1, device="cuda")
    xh, dh = to_host(x), to_host(dst)
    for op in OPS3:
        out = dst.clone()
        itr.red_rows_thread(op, x, accum=accum, out=out)
        what = f"case {case}: {rows}x{length} shift={shift} accum={accum} {op}"
        if op == "sum":
            # the thread-scope fold has a fixed order: bit for bit with the oracle's restatement
            check_exact(to_host(out), oracle.thread_rows_sum(xh, rows, length, accum, dh), what)
        else:
            check_exact(to_host(out), oracle.rows(op, xh, rows, length, accum, dh), what)


@pytest.mark.parametrize("case", range(N_CASES))
def test_rows_stats(case):
    gen = np.random.default_rng(7000 + case)
    length = int(gen.choice([1, 3, 7, 8, 16, 24, 32, 64, 65, 1024, 5000]))
    rows = int(gen.integers(1, max(2, min(5000, 2_000_000 // length))))
    shift = int(gen.choice([0, 0, 1, 3, 8]))
    x = _shifted(synth.uniform((rows * length + 8,), -4.0, 4.0, case, device="cuda"), rows * length,
                 shift).view(rows, length)
    xh = to_host(x)
    got = to_host(itr.red_rows_stats(x))
    what = f"case {case}: {rows}x{length} shift={shift}"
    s, a = oracle.rows("sum", xh, rows, length)
    check_sum(got[:, 0], s, a, what + " sum")
    check_exact(got[:, 1].copy(), oracle.rows("max", xh, rows, length), what + " max")
    check_exact(got[:, 2].copy(), oracle.rows("min", xh, rows, length), what + " min")
    check_sum(got[:, 3], a, a, what + " sum|x|")

