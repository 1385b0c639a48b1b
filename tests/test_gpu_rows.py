"""red_rows and red_rows_ragged on the GPU against the oracle: tiny and
ragged shapes (every chunk-of-8 remainder, unaligned row starts), every
lanes-per-row mapping, the split-row path for few long rows, accum, empty
rows, and the 65536 x 1024 and 2**22-ragged-row workloads at full size."""
import numpy as np
import pytest
import torch

import oracle
import int_tensor_reductions_gb300 as itr
from int_tensor_reductions_gb300 import synth
from gpu_util import check_exact, check_sum, lib_ready, to_host

pytestmark = pytest.mark.gpu

OPS = ("sum", "max", "min")


@pytest.fixture(scope="module", autouse=True)
def _lib():
    lib_ready()
    yield
    itr.red_set_knob(itr.RED_KNOB_ROWS_GROUP, 0)
    itr.red_set_knob(itr.RED_KNOB_RAGGED_GROUP, 0)
    itr.red_set_knob(itr.RED_KNOB_ROWS_ALIGNED, 0)


def _dense_case(x2d: torch.Tensor, dst: torch.Tensor, what: str):
    rows, length = x2d.shape
    xh, dh = to_host(x2d), to_host(dst)
    for accum in (False, True):
        for op in OPS:
            out = dst.clone()
            itr.red_rows(op, x2d, accum=accum, out=out)
            got = to_host(out)
            if op == "sum":
                s, a = oracle.rows("sum", xh, rows, length, accum, dh)
                check_sum(got, s, a, f"{what} sum accum={accum}")
            else:
                check_exact(got, oracle.rows(op, xh, rows, length, accum, dh), f"{what} {op} accum={accum}")


@pytest.mark.parametrize("rows,length", [
    (1, 1), (3, 7), (5, 8), (7, 9), (33, 31), (100, 40), (17, 64), (9, 1000), (4, 1024),
    (3, 5000), (300, 8191), (2, 20000), (1, 100003), (5, 300007),
])
def test_dense_shapes(rows, length):
    x = synth.uniform((rows * length + 1,), -4.0, 4.0, rows + length).cuda()
    dst = synth.uniform((rows,), -1.0, 1.0, 3).cuda()
    _dense_case(x[:rows * length].view(rows, length), dst, f"{rows}x{length}")
    # rows starting at an odd float: every row has a different head peel
    _dense_case(x[1:].view(rows, length), dst, f"{rows}x{length} shifted")


@pytest.mark.parametrize("g", [1, 2, 4, 8, 16, 32])
def test_dense_every_group_size(g):
    itr.red_set_knob(itr.RED_KNOB_ROWS_GROUP, g)
    try:
        for rows, length in ((257, 13), (130, 77), (64, 1029)):
            x = synth.normal((rows * length + 3,), g, device="cuda")
            dst = synth.uniform((rows,), -1.0, 1.0, 4, device="cuda")
            _dense_case(x[3:].view(rows, length), dst, f"G={g} {rows}x{length}")
    finally:
        itr.red_set_knob(itr.RED_KNOB_ROWS_GROUP, 0)


@pytest.mark.parametrize("aligned", [0, 2])
def test_dense_whole_block_rows_both_kernels(aligned):
    """Rows of whole 32-byte blocks from a 32-byte aligned base go to the
    aligned row kernel; knob value 2 sends the same rows to the general one.
    Both against the oracle, at every lanes-per-row setting the automatic
    choice gives for these lengths."""
    itr.red_set_knob(itr.RED_KNOB_ROWS_ALIGNED, aligned)
    try:
        for rows, length in ((3, 72), (1000, 64 + 8), (257, 256), (4099, 1024), (33, 4096), (5, 65536)):
            x = synth.normal((rows, length), rows + length, device="cuda")
            assert x.data_ptr() % 32 == 0
            dst = synth.uniform((rows,), -1.0, 1.0, 5, device="cuda")
            _dense_case(x, dst, f"aligned={aligned} {rows}x{length}")
    finally:
        itr.red_set_knob(itr.RED_KNOB_ROWS_ALIGNED, 0)


def test_dense_len0():
    x = torch.empty((5, 0), device="cuda")
    out = torch.full((5,), 2.5, device="cuda")
    itr.red_rows("sum", x, accum=True, out=out)
    assert to_host(out).tolist() == [2.5] * 5
    itr.red_rows("sum", x, out=out)
    assert to_host(out).tolist() == [0.0] * 5
    with pytest.raises(itr.RedError):
        itr.red_rows("max", x, out=out)


def test_cfg2_dense_workload():
    """65536 x 1024 normal(0,1) rows, every op, and sum with accum into a
    uniform[-1,1) dst, compared row by row in full."""
    x, dst = synth.cfg2(device="cuda")
    _dense_case(x, dst, "cfg2")


def _ragged_case(x, off, dst, what):
    xh, oh, dh = to_host(x), to_host(off), to_host(dst)
    for accum in (False, True):
        for op in OPS:
            out = dst.clone()
            itr.red_rows_ragged(op, x, off, accum=accum, out=out)
            got = to_host(out)
            if op == "sum":
                s, a = oracle.ragged("sum", xh, oh, accum, dh)
                check_sum(got, s, a, f"{what} sum accum={accum}")
            else:
                check_exact(got, oracle.ragged(op, xh, oh, accum, dh), f"{what} {op} accum={accum}")


@pytest.mark.parametrize("g", [0, 1, 2, 4, 8, 16, 32])
def test_ragged_with_empty_rows(g):
    itr.red_set_knob(itr.RED_KNOB_RAGGED_GROUP, g)
    try:
        gen = np.random.default_rng(5 + g)
        lens = gen.integers(0, 41, size=3001)
        lens[::13] = 0
        lens[7] = 300
        off = np.zeros(lens.size + 1, np.int64)
        off[1:] = np.cumsum(lens)
        x = synth.uniform((int(off[-1]),), -4.0, 4.0, 6, device="cuda")
        dst = synth.uniform((lens.size,), -1.0, 1.0, 8, device="cuda")
        _ragged_case(x, torch.from_numpy(off).cuda(), dst, f"ragged G={g}")
    finally:
        itr.red_set_knob(itr.RED_KNOB_RAGGED_GROUP, 0)


@pytest.mark.parametrize("g", [0, 1, 32])
def test_ragged_long_row_among_short_ones(g):
    """Short and empty rows around one 20000-float row and a 77-float row,
    on a base that is not 32-byte aligned."""
    itr.red_set_knob(itr.RED_KNOB_RAGGED_GROUP, g)
    try:
        gen = np.random.default_rng(40 + g)
        lens = gen.integers(0, 41, size=2000)
        lens[::11] = 0
        lens[300] = 20000
        lens[1999] = 77
        off = np.zeros(lens.size + 1, np.int64)
        off[1:] = np.cumsum(lens)
        x = synth.uniform((int(off[-1]) + 1,), -4.0, 4.0, 41, device="cuda")[1:]
        dst = synth.uniform((lens.size,), -1.0, 1.0, 42, device="cuda")
        _ragged_case(x, torch.from_numpy(off).cuda(), dst, f"G={g} long row")
    finally:
        itr.red_set_knob(itr.RED_KNOB_RAGGED_GROUP, 0)


def test_dense_short_rows_many():
    """2**17 dense rows of 1, 7 and 24 floats (one lane per row)."""
    for length in (1, 7, 24):
        rows = 1 << 17
        x = synth.uniform((rows * length + 1,), -4.0, 4.0, length, device="cuda")[1:]
        dst = synth.uniform((rows,), -1.0, 1.0, 43, device="cuda")
        _dense_case(x.view(rows, length), dst, f"{rows}x{length}")


def test_ragged_lengths_8_to_40_every_remainder():
    """One row of every length 8..40 at every start alignment 0..7."""
    lens = np.array([L for L in range(8, 41) for _ in range(8)], np.int64)
    off = np.zeros(lens.size + 1, np.int64)
    off[1:] = np.cumsum(lens)
    x = synth.uniform((int(off[-1]),), -4.0, 4.0, 10, device="cuda")
    dst = synth.uniform((lens.size,), -1.0, 1.0, 11, device="cuda")
    _ragged_case(x, torch.from_numpy(off).cuda(), dst, "lengths 8..40")


@pytest.mark.parametrize("g", [0, 1, 2, 4, 8])
def test_ragged_lengths_1_to_7_every_alignment(g):
    """Rows of 1..7 values at every start alignment 0..7 (inside one 32-byte
    block, or across one boundary), 9 rounds of them (several warps' worth)."""
    itr.red_set_knob(itr.RED_KNOB_RAGGED_GROUP, g)
    try:
        lens = np.array([L for _ in range(9) for L in range(1, 8) for _ in range(8)], np.int64)
        _ragged_case(*_ragged_from_lengths(lens, 0, 81 + g), f"G={g} lengths 1..7")
    finally:
        itr.red_set_knob(itr.RED_KNOB_RAGGED_GROUP, 0)


@pytest.mark.parametrize("mode", [1, 2])
def test_ragged_staged_and_direct_mappings(mode):
    """Both mappings of the ragged rows (1: CTA-staged tiles, 2: lanes per
    row) on short and empty rows, short rows around rows longer than the
    staged buffer (8192 floats), 8..40-value rows (a tile needs several
    staged runs) and one huge row, at two base alignments."""
    itr.red_set_knob(itr.RED_KNOB_RAGGED_STAGED, mode)
    try:
        gen = np.random.default_rng(90 + mode)
        long_among_short = gen.integers(0, 8, size=4000)
        long_among_short[[5, 1500, 1501, 3000]] = [20000, 9000, 8190, 600]
        cases = {"0..7": gen.integers(0, 8, size=5000), "long among short": long_among_short,
                 "8..40": gen.integers(8, 41, size=2100), "one huge row": np.array([200_000])}
        for name, lens in cases.items():
            for shift in (0, 3):
                _ragged_case(*_ragged_from_lengths(lens, shift, 91), f"mode={mode} {name} shift={shift}")
    finally:
        itr.red_set_knob(itr.RED_KNOB_RAGGED_STAGED, 0)


def _ragged_from_lengths(lens, shift, seed):
    off = np.zeros(len(lens) + 1, np.int64)
    off[1:] = np.cumsum(lens)
    x = synth.uniform((int(off[-1]) + 8,), -4.0, 4.0, seed, device="cuda")[shift:shift + int(off[-1])]
    dst = synth.uniform((len(lens),), -1.0, 1.0, seed + 1, device="cuda")
    return x, torch.from_numpy(off).cuda(), dst


@pytest.mark.parametrize("g", [0, 2])
@pytest.mark.parametrize("shift", range(8))
def test_ragged_every_base_alignment(g, shift):
    """1000 rows of 8..40 values (several warps' worth of rows, a ragged last
    iteration) at each of the 8 float offsets of x from a 32-byte boundary;
    the automatic lanes per row (1) and 2."""
    itr.red_set_knob(itr.RED_KNOB_RAGGED_GROUP, g)
    try:
        lens = np.random.default_rng(60 + shift).integers(8, 41, size=1000)
        _ragged_case(*_ragged_from_lengths(lens, shift, 61 + shift), f"G={g} shift={shift}")
    finally:
        itr.red_set_knob(itr.RED_KNOB_RAGGED_GROUP, 0)


@pytest.mark.parametrize("kind", ["all8", "long", "short_rows_sprinkled", "single_row", "huge_row"])
def test_ragged_shapes(kind):
    """Rows of exactly 8, rows up to 3000 values, short and empty rows
    sprinkled among 8..40-value rows, one row, and one 200000-value row, at
    two base alignments (the L2 prefetch spans round inward at both ends)."""
    gen = np.random.default_rng(70)
    if kind == "all8":
        lens = np.full(1500, 8)
    elif kind == "long":
        lens = gen.integers(8, 3000, size=700)
    elif kind == "short_rows_sprinkled":
        lens = gen.integers(8, 41, size=128 * 9 + 17)
        for t in range(0, 10, 2):
            if 128 * t + 5 < lens.size:
                lens[128 * t + 5] = t % 8
    elif kind == "single_row":
        lens = np.array([37])
    else:
        lens = np.array([200_000])
    for shift in (0, 3):
        _ragged_case(*_ragged_from_lengths(lens, shift, 71), f"{kind} shift={shift}")


def test_ragged_all_empty():
    off = torch.zeros(6, dtype=torch.int64, device="cuda")
    x = torch.empty(0, device="cuda")
    out = torch.full((5,), 1.5, device="cuda")
    itr.red_rows_ragged("max", x, off, out=out)
    assert to_host(out).tolist() == [-np.inf] * 5
    itr.red_rows_ragged("min", x, off, out=out)
    assert to_host(out).tolist() == [np.inf] * 5
    itr.red_rows_ragged("sum", x, off, out=out)
    assert to_host(out).tolist() == [0.0] * 5


def test_cfg5_ragged_workload():
    """2**22 rows of lengths 8..40, uniform[-4,4), compared row by row."""
    x, off = synth.cfg5(device="cuda")
    dst = synth.uniform((synth.CFG5_ROWS,), -1.0, 1.0, 12, device="cuda")
    _ragged_case(x, off, dst, "cfg5")
