"""red_colprod (TCOLPROD) on the GPU against the oracle: the page's 16 x 16
example with closed-form columns, the early return, the vector (8- and
4-wide) and scalar column paths with ragged column counts and unaligned
bases, row splits, int32 wrap closed forms, and both full-size workloads."""
from fractions import Fraction

import numpy as np
import pytest
import torch

import oracle
import int_tensor_reductions_gb300 as itr
from int_tensor_reductions_gb300 import synth
from conftest import golden_lines
from gpu_util import check_exact, check_prod, lib_ready, to_host

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    lib_ready()
    yield
    itr.red_set_knob(itr.RED_KNOB_COLPROD_SPLITS, 0)


def _f32_case(x: torch.Tensor, what: str, cols=None):
    R, C = x.shape
    got = to_host(itr.red_colprod(x))
    xh = to_host(x)
    if cols is not None:
        xh = np.ascontiguousarray(xh[:, cols])
        got = got[cols]
    _, pd = oracle.colprod_f32(xh, R, xh.shape[1], want_double=True)
    check_prod(got, pd, what)


def _i32_case(x: torch.Tensor, what: str):
    R, C = x.shape
    check_exact(to_host(itr.red_colprod(x)), oracle.colprod_i32(to_host(x), R, C), what)


def test_page_example_16x16():
    """pto-isa docs, "TCOLPROD", "Examples": 16 x 16 float -> 1 x 16."""
    lines = golden_lines("tcolprod_16x16.txt")
    R = int(lines[0][1])
    cs = [float(c) for _, c, _ in lines[2:]]
    exp = [Fraction(f) for _, _, f in lines[2:]]
    x = torch.tensor(cs, dtype=torch.float32, device="cuda").repeat(R, 1).contiguous()
    got = to_host(itr.red_colprod(x))
    ref = np.array([np.float32(e.numerator / e.denominator) for e in exp], np.float32)
    # Columns of +-2**k: every partial product is exact in fp32, so the GPU
    # result must be the closed form bit for bit.  The other columns round
    # in fp32 along the way: within the 5e-4 relative tolerance of the
    # exact value.
    pow2 = [j for j, c in enumerate(cs) if abs(c) in (0.25, 0.5, 1.0, 2.0, 4.0)]
    check_exact(got[pow2], ref[pow2], "16x16 closed form, power-of-two columns")
    check_prod(got, [e.numerator / e.denominator for e in exp], "16x16 closed form")


def test_early_return_leaves_out_untouched():
    """pto-isa docs, "TCOLPROD", "Constraints": R == 0 or C == 0."""
    out = torch.full((4,), 7.25, device="cuda")
    itr.red_colprod(torch.empty((0, 4), device="cuda"), out)
    torch.cuda.synchronize()
    assert to_host(out).tolist() == [7.25] * 4
    iout = torch.full((4,), -9, dtype=torch.int32, device="cuda")
    itr.red_colprod(torch.empty((0, 4), dtype=torch.int32, device="cuda"), iout)
    assert to_host(iout).tolist() == [-9] * 4
    e = torch.empty((3, 0), device="cuda")
    itr.red_colprod(e, torch.empty(0, device="cuda"))


@pytest.mark.parametrize("R,C", [(1, 1), (3, 5), (37, 129), (100, 1000), (64, 8), (5, 4),
                                 (129, 257), (1000, 96), (33, 4100), (4096, 24)])
def test_f32_shapes(R, C):
    x = synth.uniform((R * C + 2,), 0.99, 1.01, R + C).cuda()
    _f32_case(x[:R * C].view(R, C), f"{R}x{C}")
    _f32_case(x[1:R * C + 1].view(R, C), f"{R}x{C} base+1")   # scalar column path
    _f32_case(x[2:].view(R, C), f"{R}x{C} base+2")


@pytest.mark.parametrize("splits", [1, 2, 3, 7, 64])
def test_f32_forced_splits(splits):
    itr.red_set_knob(itr.RED_KNOB_COLPROD_SPLITS, splits)
    try:
        x = synth.uniform((500, 2056), 0.99, 1.01, 31, device="cuda")
        _f32_case(x, f"splits={splits}")
        xi = synth.int_choice((300, 1032), synth.INT_CHOICES, 32, device="cuda")
        _i32_case(xi, f"i32 splits={splits}")
    finally:
        itr.red_set_knob(itr.RED_KNOB_COLPROD_SPLITS, 0)


@pytest.mark.parametrize("c,R", [(1.0, 1000), (-1.0, 999), (2.0, 100), (0.5, 120), (-2.0, 37)])
def test_f32_constant_columns(c, R):
    x = torch.full((R, 40), c, dtype=torch.float32, device="cuda")
    got = to_host(itr.red_colprod(x))
    assert (got == np.float32(c ** R)).all()


def test_i32_wrap_closed_forms():
    for c, R, expected in golden_lines("tcolprod_i32_wrap.txt"):
        x = torch.full((int(R), 72), int(c), dtype=torch.int32, device="cuda")
        assert (to_host(itr.red_colprod(x)) == int(expected)).all(), (c, R)


@pytest.mark.parametrize("R,C", [(1, 3), (7, 5), (64, 8), (333, 1001), (2048, 512)])
def test_i32_shapes(R, C):
    x = synth.int_choice((R * C + 1,), synth.INT_CHOICES, R * C, device="cuda")
    _i32_case(x[:R * C].view(R, C), f"i32 {R}x{C}")
    _i32_case(x[1:].view(R, C), f"i32 {R}x{C} base+1")


def test_i32_large_values():
    g = torch.Generator(device="cuda").manual_seed(77)
    x = torch.randint(-2**31, 2**31 - 1, (129, 300), generator=g, device="cuda", dtype=torch.int64)
    _i32_case(x.to(torch.int32), "i32 full-range values")


def test_cfg4a_f32_workload():
    """4096 x 16384 uniform[0.999, 1.001]: 2048 sampled columns against the
    oracle (every column through the same kernel launch)."""
    x = synth.cfg4a(device="cuda")
    cols = np.sort(np.random.default_rng(3).choice(x.shape[1], 2048, replace=False))
    cols = np.unique(np.concatenate([cols, [0, 1, 7, 8, x.shape[1] - 1]]))
    _f32_case(x, "cfg4a", cols=cols)


def test_cfg4b_i32_workload():
    """64 x 65536 int32 from {-3..3} \\ {0}, every column bit-exact."""
    _i32_case(synth.cfg4b(device="cuda"), "cfg4b")
