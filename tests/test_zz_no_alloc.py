"""red_full_noalloc: the full reduction for callers that cannot allocate
device memory (cudaMalloc may synchronise the device, and a framework whose
allocator owns the memory may not let a library take any).  It keeps its
scratch in a fixed array inside the library.

Called through the C ABI and checked against red_full (the entry point that
uses the allocated workspace) on two calls in a row, with the tolerances of
the other tests: sums within 1e-5 * sum|x|, max / min bit for bit.  This file
is collected last so that a stop-at-first-failure run has already run every
other test; it also passes alone in a fresh process.
"""
import ctypes

import numpy as np
import pytest
import torch

import int_tensor_reductions_gb300 as itr
from int_tensor_reductions_gb300 import synth
from gpu_util import SUM_RTOL, lib_ready

pytestmark = pytest.mark.gpu

OPS = {"sum": itr.RED_SUM, "max": itr.RED_MAX, "min": itr.RED_MIN}


@pytest.fixture(scope="module", autouse=True)
def _lib():
    lib_ready()
    yield
    itr.red_set_knob(itr.RED_KNOB_FULL_CTAS_PER_SM, 0)


def _call_noalloc(op, x, out):
    stream = torch.cuda.current_stream().cuda_stream
    return itr.lib().red_full_noalloc(OPS[op], x.data_ptr(), x.numel(), out.data_ptr(), stream)


@pytest.mark.parametrize("n", [1, 7, 32, 1000, 65537, 1 << 20, (1 << 26) + 3])
def test_matches_red_full_on_two_calls(n):
    x = synth.uniform((n + 1,), -1.0, 1.0, n % 997, device="cuda")[1:]
    scale = float(x.double().abs().sum())
    for op in OPS:
        ref = float(itr.red_full(op, x)[0])
        for call in range(2):
            out = torch.full((1,), float("nan"), device="cuda")
            assert _call_noalloc(op, x, out) == itr.RED_OK, itr.red_last_error()
            got = float(out[0])
            if op == "sum":
                assert abs(got - ref) <= SUM_RTOL * scale, (n, call, got, ref)
            else:
                assert np.float32(got).view(np.uint32) == np.float32(ref).view(np.uint32), (n, op, call)


def test_empty_input():
    out = torch.full((1,), 5.0, device="cuda")
    e = torch.empty(0, device="cuda")
    assert _call_noalloc("sum", e, out) == itr.RED_OK
    assert float(out[0]) == 0.0
    assert _call_noalloc("max", e, out) == itr.RED_EINVAL


def test_rejects_more_ctas_than_the_scratch_holds():
    x = synth.uniform((1 << 26,), -1.0, 1.0, 3, device="cuda")
    out = torch.zeros(1, device="cuda")
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    per_sm = 32
    if sms * per_sm <= 4096:
        pytest.skip("this GPU cannot ask for more CTAs than the scratch holds")
    itr.red_set_knob(itr.RED_KNOB_FULL_CTAS_PER_SM, per_sm)
    try:
        assert _call_noalloc("sum", x, out) == itr.RED_EINVAL
        assert "static scratch" in itr.red_last_error()
    finally:
        itr.red_set_knob(itr.RED_KNOB_FULL_CTAS_PER_SM, 0)
    assert _call_noalloc("sum", x, out) == itr.RED_OK
