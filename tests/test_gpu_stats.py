"""red_full_stats (sum, max, min and sum |x| from one read) on the GPU against
the oracle: every length 1..96 at unaligned starts, multi-CTA sizes with
ragged tails, and the 2**30-element vector."""
import numpy as np
import pytest
import torch

import oracle
import int_tensor_reductions_gb300 as itr
from int_tensor_reductions_gb300 import synth
from gpu_util import SUM_RTOL, check_exact, check_sum, lib_ready, to_host

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    lib_ready()


def _check(xd: torch.Tensor, what: str):
    xh = to_host(xd)
    s, a = oracle.full_sum(xh)
    got = to_host(itr.red_full_stats(xd))
    check_sum(got[0:1], s, a, what + " sum")
    check_exact(got[1:2], np.array([oracle.full_max(xh)], np.float32), what + " max")
    check_exact(got[2:3], np.array([oracle.full_min(xh)], np.float32), what + " min")
    # sum |x|: a sum of non-negative terms, so its own scale is the bound
    check_sum(got[3:4], a, a, what + " sum|x|")


def test_every_small_length():
    base = synth.uniform((200,), -1.0, 1.0, 21).cuda()
    for n in range(1, 97):
        for shift in (0, 3):
            _check(base[shift:shift + n], f"n={n} shift={shift}")


@pytest.mark.parametrize("n", [4097, 1_000_003, synth.CFG1_N, (1 << 24) + 7])
def test_multi_cta_sizes(n):
    x = synth.normal((n + 1,), n % 101, device="cuda")
    _check(x[:n], f"n={n}")
    _check(x[1:], f"n={n} shifted")


def test_agrees_with_separate_calls():
    x = synth.normal((3_000_001,), 5, device="cuda")
    got = to_host(itr.red_full_stats(x))
    assert got[1] == float(itr.red_full("max", x)[0])
    assert got[2] == float(itr.red_full("min", x)[0])
    s = float(itr.red_full("sum", x)[0])
    assert abs(got[0] - s) <= 2 * SUM_RTOL * float(got[3])


def test_empty_rejected():
    with pytest.raises(itr.RedError):
        itr.red_full_stats(torch.empty(0, device="cuda"))


def test_cfg3_4gib_vector():
    x = synth.cfg3(device="cuda")
    _check(x, "cfg3")
    del x
    torch.cuda.empty_cache()


def _check_rows(x2d: torch.Tensor, what: str):
    rows, length = x2d.shape
    xh = to_host(x2d)
    got = to_host(itr.red_rows_stats(x2d))
    s, a = oracle.rows("sum", xh, rows, length)
    check_sum(got[:, 0], s, a, what + " sum")
    check_exact(got[:, 1].copy(), oracle.rows("max", xh, rows, length), what + " max")
    check_exact(got[:, 2].copy(), oracle.rows("min", xh, rows, length), what + " min")
    check_sum(got[:, 3], a, a, what + " sum|x|")


@pytest.mark.parametrize("rows,length", [(1, 1), (5, 7), (33, 8), (100, 24), (257, 41), (64, 1024), (9, 5000),
                                         (300, 3), (1000, 5), (1, 16), (3, 16), (4099, 16), (17, 32),
                                         (2049, 32), (1000, 64), (33, 64)])
def test_rows_stats_shapes(rows, length):
    x = synth.uniform((rows * length + 3,), -4.0, 4.0, rows + length, device="cuda")
    _check_rows(x[:rows * length].view(rows, length), f"{rows}x{length}")
    _check_rows(x[3:].view(rows, length), f"{rows}x{length} shifted")


def test_rows_stats_workload():
    x, _ = synth.cfg2(device="cuda")
    _check_rows(x, "65536x1024")


def test_rows_stats_rejects_empty_rows():
    with pytest.raises(itr.RedError):
        itr.red_rows_stats(torch.empty((3, 0), device="cuda"))
