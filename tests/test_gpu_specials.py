"""Special values, which the synthetic workloads never contain: infinities
propagate as in IEEE arithmetic, a column product of 0 and inf is NaN, and
the packed flush-to-zero sum of Apache TVM docs, "reduction ->
sm100_packed", "Generated CUDA" (add.rn.ftz.f32x2) flushes denormal inputs,
so a sum of denormals is 0 while max / min return them exactly."""
import math

import numpy as np
import pytest
import torch

import int_tensor_reductions_gb300 as itr
from int_tensor_reductions_gb300 import synth
from gpu_util import lib_ready, to_host

pytestmark = pytest.mark.gpu

INF = float("inf")
DENORM = 2.0**-140  # below FLT_MIN (2**-126), exactly representable


@pytest.fixture(scope="module", autouse=True)
def _lib():
    lib_ready()


@pytest.mark.parametrize("n", [5, 1000, 1_000_003])
def test_full_with_infinities(n):
    x = synth.uniform((n,), -1.0, 1.0, n, device="cuda")
    finite_min = float(x.min())
    x[n // 2] = INF
    assert float(itr.red_full("sum", x)[0]) == INF
    assert float(itr.red_full("max", x)[0]) == INF
    assert float(itr.red_full("min", x)[0]) == finite_min
    st = to_host(itr.red_full_stats(x))
    assert st[0] == INF and st[1] == INF and st[2] == finite_min and st[3] == INF
    x[n - 1] = -INF
    assert float(itr.red_full("min", x)[0]) == -INF
    assert math.isnan(float(itr.red_full("sum", x)[0]))  # inf + (-inf)


def test_rows_ragged_and_cols_with_infinities():
    x = synth.uniform((300, 77), -1.0, 1.0, 3, device="cuda")
    x[5, 7] = INF
    x[9, 0] = -INF
    s = to_host(itr.red_rows("sum", x))
    assert s[5] == INF and s[9] == -INF and np.isfinite(np.delete(s, [5, 9])).all()
    m = to_host(itr.red_rows("max", x))
    assert m[5] == INF
    off = torch.arange(0, 300 * 77 + 1, 77, dtype=torch.int64, device="cuda")
    rg = to_host(itr.red_rows_ragged("sum", x.view(-1), off))
    assert rg[5] == INF and rg[9] == -INF
    fin = np.delete(np.arange(300), [5, 9])
    assert np.allclose(rg[fin], s[fin], rtol=0, atol=1e-4)
    c = to_host(itr.red_cols("sum", x))
    assert c[7] == INF and c[0] == -INF
    p = torch.full((40, 24), 1.0, device="cuda")
    p[3, 2] = INF
    p[4, 5] = INF
    p[6, 5] = 0.0
    pr = to_host(itr.red_colprod(p))
    assert pr[2] == INF and math.isnan(pr[5]) and (np.delete(pr, [2, 5]) == 1.0).all()


def test_typed_half_and_bf16_infinities():
    for dt in (torch.float16, torch.bfloat16):
        x = torch.full((4096,), 0.5, dtype=dt, device="cuda")
        x[4000] = INF
        assert float(itr.red_full_typed("sum", x)[0]) == INF
        assert float(itr.red_full_typed("max", x)[0]) == INF
        assert float(itr.red_full_typed("min", x)[0]) == 0.5


@pytest.mark.parametrize("n", [7, 8, 33, 100_000])
def test_denormals_flush_in_sums_and_stay_in_max_min(n):
    x = torch.full((n,), DENORM, dtype=torch.float32, device="cuda")
    x[n // 3] = 2 * DENORM
    x[0] = -DENORM
    assert float(itr.red_full("sum", x)[0]) == 0.0
    assert float(itr.red_full("max", x)[0]) == 2 * DENORM
    assert float(itr.red_full("min", x)[0]) == -DENORM
    rows = to_host(itr.red_rows("max", x.view(1, n)))
    assert rows[0] == 2 * DENORM
