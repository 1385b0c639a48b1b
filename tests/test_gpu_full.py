"""red_full on the GPU against the oracle: every length 1..96 (all head and
tail remainders), multi-CTA sizes with ragged tails, unaligned starts, every
grid stage, and the 4 GiB workload in the benchmark's launch configuration."""
import numpy as np
import pytest
import torch

import oracle
import int_tensor_reductions_gb300 as itr
from int_tensor_reductions_gb300 import synth
from conftest import golden_lines
from gpu_util import check_exact, check_sum, lib_ready, to_host

pytestmark = pytest.mark.gpu

MODES = [itr.RED_MODE_TWO_PASS, itr.RED_MODE_LAST_BLOCK, itr.RED_MODE_ATOMIC]


@pytest.fixture(scope="module", autouse=True)
def _lib():
    lib_ready()
    yield
    itr.red_set_full_mode(itr.RED_MODE_AUTO)


def _check_all_ops(xd: torch.Tensor, what: str):
    xh = to_host(xd)
    s, a = oracle.full_sum(xh)
    check_sum(to_host(itr.red_full("sum", xd)), s, a, what + " sum")
    check_exact(to_host(itr.red_full("max", xd)), np.array([oracle.full_max(xh)], np.float32), what + " max")
    check_exact(to_host(itr.red_full("min", xd)), np.array([oracle.full_min(xh)], np.float32), what + " min")


def test_page_demo_sum32():
    """Apache TVM docs, "reduction -> sm100_packed": B == sum(A), 32 floats."""
    rows = dict((r[0], r[1:]) for r in golden_lines("sm100_packed_demo_sum32.txt"))
    a = torch.tensor([float(v) for v in rows["A"]], dtype=torch.float32, device="cuda")
    for m in MODES:
        itr.red_set_full_mode(m)
        assert float(itr.red_full("sum", a)[0]) == float(rows["B"][0])


@pytest.mark.parametrize("mode", MODES)
def test_every_small_length(mode):
    itr.red_set_full_mode(mode)
    base = synth.uniform((200,), -1.0, 1.0, 7).cuda()
    for n in range(1, 97):
        for shift in (0, 1, 3, 5):  # unaligned starts peel a head of 1..7
            _check_all_ops(base[shift:shift + n], f"n={n} shift={shift}")


@pytest.mark.parametrize("mode", MODES)
@pytest.mark.parametrize("n", [1000, 65537, 1_000_003, synth.CFG1_N, (1 << 24) + 5])
def test_multi_cta_sizes(mode, n):
    itr.red_set_full_mode(mode)
    x = synth.uniform((n + 3,), -1.0, 1.0, n % 1000, device="cuda")
    _check_all_ops(x[:n], f"n={n}")
    _check_all_ops(x[3:], f"n={n} shifted")


def test_extremes_at_every_position_of_a_tail():
    """Plant the extreme in the head, interior and tail of a multi-CTA vector."""
    n = 3 * 2**20 + 7
    x = synth.uniform((n + 1,), -1.0, 1.0, 9, device="cuda")[1:]
    for p in (0, 1, 6, 7, 8, n // 2, n - 8, n - 7, n - 1):
        y = x.clone()
        y[p] = 5.0
        assert float(itr.red_full("max", y)[0]) == 5.0
        y[p] = -5.0
        assert float(itr.red_full("min", y)[0]) == -5.0


def test_sum_closed_form_arange():
    for n in (33, 4096, 1 << 20):
        x = torch.arange(n, dtype=torch.float32, device="cuda")
        # exact partial sums need n(n-1)/2 < 2**24 for every order; check
        # against the tolerance otherwise
        got = float(itr.red_full("sum", x)[0])
        exact = n * (n - 1) / 2
        assert abs(got - exact) <= 1e-5 * exact


def test_empty():
    out = torch.full((1,), 3.0, device="cuda")
    itr.red_full("sum", torch.empty(0, device="cuda"), out)
    assert float(out[0]) == 0.0
    with pytest.raises(itr.RedError):
        itr.red_full("max", torch.empty(0, device="cuda"), out)


def test_cfg1_vector():
    x = synth.cfg1(device="cuda")
    for m in MODES:
        itr.red_set_full_mode(m)
        _check_all_ops(x, f"cfg1 mode {m}")


@pytest.fixture(scope="module")
def cfg3():
    """The 2**30-element normal(0,1) vector and its oracle results."""
    x = synth.cfg3(device="cuda")
    xh = to_host(x)
    ref = {"sum": oracle.full_sum(xh), "max": oracle.full_max(xh), "min": oracle.full_min(xh)}
    del xh
    yield x, ref
    del x
    torch.cuda.empty_cache()


@pytest.mark.parametrize("mode", MODES)
def test_cfg3_4gib_vector(cfg3, mode):
    """The 4 GiB workload in the launch configuration the benchmark times."""
    x, ref = cfg3
    itr.red_set_full_mode(mode)
    s, a = ref["sum"]
    check_sum(to_host(itr.red_full("sum", x)), s, a, f"cfg3 sum mode {mode}")
    check_exact(to_host(itr.red_full("max", x)), np.array([ref["max"]], np.float32), "cfg3 max")
    check_exact(to_host(itr.red_full("min", x)), np.array([ref["min"]], np.float32), "cfg3 min")


def test_binding_rejects_short_buffers():
    """The Python wrappers check buffer sizes the C ABI cannot see (it takes
    plain pointers): an empty out, or offsets without rows + 1 entries, is a
    ValueError before anything is launched."""
    x = torch.ones(100, device="cuda")
    e = torch.empty(0, device="cuda")
    for call in (lambda: itr.red_full("sum", x, e), lambda: itr.red_full_noalloc("sum", x, e),
                 lambda: itr.red_full_typed("sum", x, e), lambda: itr.red_full_stats(x, torch.empty(3, device="cuda")),
                 lambda: itr.red_rows_ragged("sum", x, torch.empty(0, dtype=torch.int64, device="cuda")),
                 lambda: itr.red_rows("sum", x.view(10, 10), out=torch.empty(9, device="cuda"))):
        with pytest.raises(ValueError):
            call()
