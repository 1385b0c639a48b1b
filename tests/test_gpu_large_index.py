"""Inputs of more than 2**31 elements, so that any 32-bit index or offset
arithmetic would read or write the wrong place.  Values are ones with a few
markers placed beyond element 2**31; every expected value is a closed form
(no host copy of the 8+ GiB inputs): integer-valued sums below 2**24 per
partial are exact in fp32, and max / min are exact."""
import numpy as np
import pytest
import torch

import int_tensor_reductions_gb300 as itr
from gpu_util import lib_ready, to_host

pytestmark = pytest.mark.gpu

BIG = (1 << 31) + 37


@pytest.fixture(scope="module", autouse=True)
def _lib():
    lib_ready()


@pytest.fixture(autouse=True)
def _free():
    yield
    torch.cuda.empty_cache()


def test_full_beyond_2p31():
    x = torch.ones(BIG, device="cuda")
    x[BIG - 1] = 1.0e6
    x[(1 << 31) + 3] = -5.0e5
    assert float(itr.red_full("max", x)[0]) == 1.0e6
    assert float(itr.red_full("min", x)[0]) == -5.0e5
    exact = (BIG - 2) + 1.0e6 - 5.0e5
    s = float(itr.red_full("sum", x)[0])
    assert abs(s - exact) <= 1e-5 * (BIG - 2 + 1.5e6)
    st = to_host(itr.red_full_stats(x))
    assert st[1] == 1.0e6 and st[2] == -5.0e5
    assert abs(st[0] - exact) <= 1e-5 * (BIG - 2 + 1.5e6)
    assert abs(st[3] - (BIG - 2 + 1.5e6)) <= 1e-5 * (BIG - 2 + 1.5e6)


def test_dense_rows_beyond_2p31():
    """2**21 rows of 1025: row r starts at element r * 1025, past 2**31 for
    the last rows (one warp per row)."""
    rows, length = 1 << 21, 1025
    x = torch.ones((rows, length), device="cuda")
    x[rows - 1, 7] = 100.0
    x[rows - 2, 1024] = -3.0
    s = to_host(itr.red_rows("sum", x))
    want = np.full(rows, float(length))
    want[rows - 1] += 99.0
    want[rows - 2] -= 4.0
    assert np.array_equal(s.astype(np.float64), want)
    m = to_host(itr.red_rows("max", x))
    assert m[rows - 1] == 100.0 and (m[:rows - 1] == 1.0).all()


def test_split_rows_beyond_2p31():
    """3 rows of 2**30 + 5 (the several-CTAs-per-row path)."""
    rows, length = 3, (1 << 30) + 5
    x = torch.ones((rows, length), device="cuda")
    x[2, length - 1] = 7.0
    m = to_host(itr.red_rows("max", x))
    assert m.tolist() == [1.0, 1.0, 7.0]
    s = to_host(itr.red_rows("sum", x)).astype(np.float64)
    want = np.array([length, length, length + 6.0])
    assert (np.abs(s - want) <= 1e-5 * want).all()


def test_ragged_beyond_2p31():
    """2**22 ragged rows of 500..1000 values (more than 2**31 values in all):
    with ones the row sums are the row lengths."""
    g = torch.Generator(device="cuda")
    g.manual_seed(9)
    lens = torch.randint(500, 1001, (1 << 22,), generator=g, device="cuda", dtype=torch.int64)
    off = torch.zeros((1 << 22) + 1, dtype=torch.int64, device="cuda")
    torch.cumsum(lens, 0, out=off[1:])
    nnz = int(off[-1].item())
    assert nnz > (1 << 31)
    x = torch.ones(nnz, device="cuda")
    x[nnz - 2] = 9.0
    s = itr.red_rows_ragged("sum", x, off)
    want = lens.to(torch.float32)
    want[-1] += 8.0
    assert torch.equal(s, want)
    m = to_host(itr.red_rows_ragged("max", x, off))
    assert m[-1] == 9.0 and (m[:-1] == 1.0).all()


def test_cols_beyond_2p31():
    """A (2**16 + 3) x (2**15 + 16) column sum: the last rows start past
    element 2**31."""
    R, C = (1 << 16) + 3, (1 << 15) + 16
    x = torch.ones((R, C), device="cuda")
    x[R - 1, C - 1] = 5.0
    s = to_host(itr.red_cols("sum", x)).astype(np.float64)
    want = np.full(C, float(R))
    want[C - 1] += 4.0
    assert np.array_equal(s, want)


def test_typed_half_max_beyond_2p31():
    x = torch.ones(BIG, dtype=torch.float16, device="cuda")
    x[BIG - 5] = 3.5
    x[(1 << 31) + 1] = -2.0
    assert float(itr.red_full_typed("max", x)[0]) == 3.5
    assert float(itr.red_full_typed("min", x)[0]) == -2.0


def test_cols_16bit_beyond_2p31():
    """A (2**16 + 3) x (2**15 + 16) bfloat16 column max (128-bit loads, 8 rows
    in flight per lane): zeros with markers in rows whose elements lie past
    2**31."""
    R, C = (1 << 16) + 3, (1 << 15) + 16
    x = torch.zeros((R, C), dtype=torch.bfloat16, device="cuda")
    x[R - 1, C - 1] = 5.0
    x[R - 2, 7] = 3.0
    x[(1 << 31) // C + 1, 100] = 2.0
    m = itr.red_cols("max", x).to(torch.float64).cpu().numpy()
    want = np.zeros(C)
    want[C - 1], want[7], want[100] = 5.0, 3.0, 2.0
    assert np.array_equal(m, want)


def test_typed_short_rows_beyond_2p31():
    """2**28 + 3 uint16 rows of 8 (two rows per 32-byte block, the last row
    after the last whole block): markers in rows past element 2**31."""
    rows = (1 << 28) + 3
    x = torch.zeros((rows, 8), dtype=torch.int16, device="cuda")
    marks = {rows - 1: 7, rows - 2: 9, (1 << 28) + 0: 11, (1 << 28) - 1: 13}
    for r, v in marks.items():
        x[r, 5] = v
    out = itr.red_rows_typed("max", x, dtype="u16")
    assert int((out != 0).sum()) == len(marks)
    for r, v in marks.items():
        assert int(out[r]) == v, r
