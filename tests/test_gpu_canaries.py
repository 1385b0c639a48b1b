"""No entry point writes outside its output.  Each output is a slice of a
larger buffer whose padding on both sides holds a sentinel bit pattern; after
the call the padding must be unchanged.  Shapes include one element, ragged
tails, unaligned bases and multi-CTA sizes; every grid stage of the full
reduction and forced row splits of the column reductions are covered."""
import numpy as np
import pytest
import torch

import int_tensor_reductions_gb300 as itr
from int_tensor_reductions_gb300 import synth
from gpu_util import lib_ready

pytestmark = pytest.mark.gpu

PAD = 64  # elements of padding on each side
SENTINEL32 = 0x7FC0DEAD  # a NaN payload no reduction of finite data produces
SENTINEL16 = 0x7E5A


@pytest.fixture(scope="module", autouse=True)
def _lib():
    lib_ready()


def _guarded(n, dtype, shift=0):
    """(buffer, view): a view of n elements at offset PAD + shift."""
    esz = torch.empty(0, dtype=dtype).element_size()
    bits = torch.int32 if esz == 4 else torch.int16
    buf = torch.full((2 * PAD + n + shift,), SENTINEL32 if esz == 4 else SENTINEL16, dtype=torch.int64,
                     device="cuda").to(bits).view(dtype)
    return buf, buf[PAD + shift:PAD + shift + n]


def _intact(buf, n, shift, what):
    torch.cuda.synchronize()
    raw = buf.view(torch.int32 if buf.element_size() == 4 else torch.int16).cpu().numpy()
    want = np.int64(SENTINEL32 if buf.element_size() == 4 else SENTINEL16)
    want = want.astype(raw.dtype)
    head, tail = raw[:PAD + shift], raw[PAD + shift + n:]
    assert (head == want).all() and (tail == want).all(), f"{what}: write outside the output"


@pytest.mark.parametrize("mode", [itr.RED_MODE_AUTO, itr.RED_MODE_TWO_PASS, itr.RED_MODE_LAST_BLOCK,
                                  itr.RED_MODE_ATOMIC])
def test_full_and_stats(mode):
    itr.red_set_full_mode(mode)
    try:
        for n in (1, 9, 100_003, 5_000_001):
            x = synth.uniform((n + 1,), -1.0, 1.0, n, device="cuda")[1:]
            for op in ("sum", "max", "min"):
                buf, out = _guarded(1, torch.float32, shift=n % 3)
                itr.red_full(op, x, out)
                _intact(buf, 1, n % 3, f"red_full {op} n={n}")
            buf, out = _guarded(4, torch.float32)
            itr.red_full_stats(x, out)
            _intact(buf, 4, 0, f"red_full_stats n={n}")
    finally:
        itr.red_set_full_mode(itr.RED_MODE_AUTO)


def test_full_noalloc():
    x = synth.uniform((1_000_003,), -1.0, 1.0, 3, device="cuda")
    for op in ("sum", "max", "min"):
        buf, out = _guarded(1, torch.float32)
        itr.red_full_noalloc(op, x, out)
        _intact(buf, 1, 0, f"red_full_noalloc {op}")


@pytest.mark.parametrize("rows,length", [(1, 1), (3, 7), (257, 41), (1000, 1024), (5, 100_000)])
def test_rows_thread_stats(rows, length):
    x = synth.uniform((rows * length + 1,), -1.0, 1.0, rows, device="cuda")[1:].view(rows, length)
    for op in ("sum", "max", "min"):
        for accum in (False, True):
            buf, out = _guarded(rows, torch.float32, shift=1)
            out.fill_(0.5)
            itr.red_rows(op, x, accum=accum, out=out)
            _intact(buf, rows, 1, f"red_rows {op} {rows}x{length} accum={accum}")
        if length <= 64:
            buf, out = _guarded(rows, torch.float32)
            itr.red_rows_thread(op, x, out=out)
            _intact(buf, rows, 0, f"red_rows_thread {op} {rows}x{length}")
    buf, out = _guarded(4 * rows, torch.float32)
    itr.red_rows_stats(x, out.view(rows, 4))
    _intact(buf, 4 * rows, 0, f"red_rows_stats {rows}x{length}")


@pytest.mark.parametrize("mode", [0, 1, 2])
def test_ragged_invalid_offsets_stay_inside(mode):
    """Offsets that decrease, go negative or pass nnz (results unspecified,
    the call succeeds): x is a slice of a sentinel-padded buffer, and
    neither the padding around out nor any value beyond x may show up; both
    mappings (staged tiles, lanes per row) and the automatic choice."""
    itr.red_set_knob(itr.RED_KNOB_RAGGED_STAGED, mode)
    try:
        nnz = 3000
        xbuf = torch.full((nnz + 2 * PAD,), 1e30, device="cuda")
        x = xbuf[PAD:PAD + nnz]
        x.copy_(synth.uniform((nnz,), -1.0, 1.0, 5, device="cuda"))
        gen = np.random.default_rng(7)
        off = np.cumsum(gen.integers(0, 6, size=1201)).astype(np.int64)
        off[100:110] = off[100:110][::-1].copy()  # decreasing pairs
        off[300] = -50
        off[500] = nnz + 1000
        off[900:] += 2 * nnz  # past the end
        offd = torch.from_numpy(off).cuda()
        for op in ("sum", "max", "min"):
            buf, out = _guarded(off.size - 1, torch.float32, shift=1)
            itr.red_rows_ragged(op, x, offd, out=out)
            _intact(buf, off.size - 1, 1, f"red_rows_ragged {op} mode={mode} invalid offsets")
            got = out.cpu().numpy()
            finite = got[np.isfinite(got)]
            assert (np.abs(finite) < 1e29).all(), "a value from outside x was read"
    finally:
        itr.red_set_knob(itr.RED_KNOB_RAGGED_STAGED, 0)


def test_ragged_with_empty_rows():
    lens = np.random.default_rng(3).integers(0, 41, size=2001)
    lens[::7] = 0
    off = np.zeros(lens.size + 1, np.int64)
    off[1:] = np.cumsum(lens)
    x = synth.uniform((int(off[-1]),), -1.0, 1.0, 4, device="cuda")
    offd = torch.from_numpy(off).cuda()
    for op in ("sum", "max", "min"):
        buf, out = _guarded(lens.size, torch.float32, shift=2)
        itr.red_rows_ragged(op, x, offd, out=out)
        _intact(buf, lens.size, 2, f"red_rows_ragged {op}")


@pytest.mark.parametrize("splits", [0, 1, 3])
@pytest.mark.parametrize("dtype", ["f32", "i32", "f16", "u16"])
def test_cols_and_typed(dtype, splits):
    itr.red_set_knob(itr.RED_KNOB_COLPROD_SPLITS, splits)
    try:
        for R, C in ((1, 1), (37, 129), (700, 1040), (64, 4100)):
            for op in ("sum", "max", "prod"):
                x = synth.col_input(op, dtype, (R, C), R + C, device="cuda")
                buf, out = _guarded(C, x.dtype, shift=1)
                itr.red_cols(op, x, out, dtype=dtype)
                _intact(buf, C, 1, f"red_cols {op} {dtype} {R}x{C}")
                buf, out = _guarded(R, x.dtype)
                itr.red_rows_typed(op, x, out=out, dtype=dtype)
                _intact(buf, R, 0, f"red_rows_typed {op} {dtype} {R}x{C}")
                buf, out = _guarded(1, x.dtype)
                itr.red_full_typed(op, x, out, dtype=dtype)
                _intact(buf, 1, 0, f"red_full_typed {op} {dtype} {R}x{C}")
    finally:
        itr.red_set_knob(itr.RED_KNOB_COLPROD_SPLITS, 0)


@pytest.mark.parametrize("dtype", ["f32", "f16", "i32"])
def test_cols_valid_region_of_wider_rows(dtype):
    """Column reductions of the R x C valid region of rows ld > C apart:
    nothing is written past out[C - 1], whatever vector width ld allows."""
    for R, C, ld in ((37, 100, 104), (9, 12, 16), (64, 1000, 1024), (5, 3, 64), (300, 24, 40)):
        for op in ("sum", "prod"):
            full = synth.col_input(op, dtype, (R, ld), R + C, device="cuda")
            buf, out = _guarded(C, full.dtype)
            itr.red_cols(op, full[:, :C], out, dtype=dtype)
            _intact(buf, C, 0, f"red_cols {op} {dtype} {R}x{C} ld={ld}")

