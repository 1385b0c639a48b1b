"""red_rows_thread and the device header red_device.cuh (the sm100_packed
thread-scope fold) on the GPU: sums bit for bit against the oracle that takes
the page's steps in its order, for every length 1..64 (all chunk remainders),
with and without accum; max / min bit for bit against the plain oracle; the
hand-worked rounding-order cases and the page's 32-element demonstration."""
import numpy as np
import pytest
import torch

import oracle
import int_tensor_reductions_gb300 as itr
from int_tensor_reductions_gb300 import synth
from conftest import golden_lines
from gpu_util import check_exact, lib_ready, to_host

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    lib_ready()


def test_page_demo_sum32():
    """Apache TVM docs, "reduction -> sm100_packed", "Demonstration program":
    one thread sums 32 floats, B == sum(A)."""
    a = torch.arange(32, dtype=torch.float32, device="cuda").view(1, 32)
    assert float(itr.red_rows_thread("sum", a)[0]) == 496.0


def test_hand_worked_rounding_order():
    for name, accum, dst, expected, *vals in golden_lines("sm100_packed_fold_order.txt"):
        a = torch.tensor([[float(v) for v in vals]], dtype=torch.float32, device="cuda")
        out = torch.full((1,), float(dst), device="cuda")
        itr.red_rows_thread("sum", a, accum=bool(int(accum)), out=out)
        assert float(out[0]) == float(expected), name


@pytest.mark.parametrize("shift", [0, 1])
@pytest.mark.parametrize("length", list(range(1, 65)))
def test_every_length_bit_exact(length, shift):
    """300 rows (two CTAs of 128 and a partial third); shift 0 stages the
    32-byte aligned tiles with 256-bit loads, shift 1 (base 4 bytes past a
    boundary) with the scalar loop."""
    rows = 300
    x = synth.uniform((rows * length + 1,), -4.0, 4.0, length, device="cuda")[shift:shift + rows * length]
    x = x.view(rows, length)
    dst = synth.uniform((rows,), -1.0, 1.0, 100 + length, device="cuda")
    xh, dh = to_host(x), to_host(dst)
    for accum in (False, True):
        out = dst.clone()
        itr.red_rows_thread("sum", x, accum=accum, out=out)
        check_exact(to_host(out), oracle.thread_rows_sum(xh, rows, length, accum, dh), f"len={length} sum")
        for op in ("max", "min"):
            out = dst.clone()
            itr.red_rows_thread(op, x, accum=accum, out=out)
            check_exact(to_host(out), oracle.rows(op, xh, rows, length, accum, dh), f"len={length} {op}")


def test_many_rows_matches_oracle_and_red_rows():
    """2**16 rows of 32 (the page's length) across many CTAs: sums bit-exact
    to the page order and within tolerance of red_rows."""
    rows, length = 1 << 16, 32
    x = synth.normal((rows, length), 3, device="cuda")
    got = to_host(itr.red_rows_thread("sum", x))
    check_exact(got, oracle.thread_rows_sum(to_host(x), rows, length), "2^16 x 32 sum")
    ref = to_host(itr.red_rows("sum", x)).astype(np.float64)
    scale = to_host(x.abs().sum(1)).astype(np.float64)
    assert (np.abs(got - ref) <= 2e-5 * scale).all()


def test_rejects_bad_lengths():
    with pytest.raises(itr.RedError):
        itr.red_rows_thread("sum", torch.ones((4, 65), device="cuda"))
    with pytest.raises(itr.RedError):
        itr.red_rows_thread("sum", torch.ones((4, 0), device="cuda"))
