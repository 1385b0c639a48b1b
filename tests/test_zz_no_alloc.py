"""red_full_noalloc: the full reduction for callers that cannot allocate
device memory (cudaMalloc may synchronise the device, and a framework whose
allocator owns the memory may not let a library take any).  It keeps its
scratch in a fixed array inside the library.

Called through the C ABI and checked against the oracle (sums within
1e-5 * sum|x|, max / min bit for bit, the tolerances of every other test) on
two calls in a row, the second of which finds the first call's contents in
the shared scratch; the sizes include the 2^30-element vector of the large
full-reduction workload, whose launch uses one partial slot per resident CTA.
Its results also agree with red_full's within the same tolerance.  This file
is collected last so that a stop-at-first-failure run has already run every
other test; it also passes alone in a fresh process.
"""
import numpy as np
import pytest
import torch

import int_tensor_reductions_gb300 as itr
import oracle
from int_tensor_reductions_gb300 import synth
from gpu_util import SUM_RTOL, check_exact, lib_ready, to_host

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


def _two_calls(x, h, what):
    for op in OPS:
        want = oracle.full(op, h)  # sum: (exact sum, sum|x|); max / min: float32
        ref = to_host(itr.red_full(op, x))[0]
        for call in range(2):
            out = torch.full((1,), float("nan"), device="cuda")
            assert _call_noalloc(op, x, out) == itr.RED_OK, itr.red_last_error()
            got = to_host(out)[0]
            if op == "sum":
                exact, abs_sum = want
                assert abs(float(got) - exact) <= SUM_RTOL * abs_sum, (what, call, float(got), exact)
                assert abs(float(got) - float(ref)) <= 2 * SUM_RTOL * abs_sum, (what, call, float(got), float(ref))
            else:
                check_exact(np.float32(got), want, f"{what} {op} call {call}")
                check_exact(np.float32(got), ref, f"{what} {op} call {call} vs red_full")


@pytest.mark.parametrize("n", [1, 7, 32, 1000, 65537, 1 << 20, (1 << 26) + 3])
def test_matches_the_oracle_on_two_calls(n):
    # one element of offset: x starts 4 bytes past a 32-byte boundary
    x = synth.uniform((n + 1,), -1.0, 1.0, n % 997, device="cuda")[1:]
    _two_calls(x, to_host(x), f"n={n}")


def test_large_vector_on_two_calls():
    """The 2^30-element N(0,1) vector of the large full-reduction workload
    (4 GiB): every resident CTA of the launch writes a partial slot."""
    x = synth.cfg3("cuda")
    _two_calls(x, to_host(x), "2^30")
    del x
    torch.cuda.empty_cache()


def test_empty_input():
    out = torch.full((1,), 5.0, device="cuda")
    e = torch.empty(0, device="cuda")
    assert _call_noalloc("sum", e, out) == itr.RED_OK
    assert float(out[0]) == 0.0
    assert _call_noalloc("max", e, out) == itr.RED_EINVAL


def test_rejects_more_ctas_than_the_scratch_holds():
    """A launch asking for more CTAs than the scratch has partial slots is
    refused before anything runs.  The vector (2^28 floats) is long enough
    that its CTA count is the knob's (32 per SM), not the data's: it would
    give every thread of 16384 512-thread CTAs 32 floats."""
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    per_sm = 32
    if sms * per_sm <= 4096:
        pytest.skip("this GPU cannot ask for more CTAs than the scratch holds")
    x = torch.empty(1 << 28, device="cuda")  # contents unused: the call is refused on the host
    out = torch.zeros(1, device="cuda")
    itr.red_set_knob(itr.RED_KNOB_FULL_CTAS_PER_SM, per_sm)
    try:
        assert _call_noalloc("sum", x, out) == itr.RED_EINVAL
        msg = itr.red_last_error()
        assert "static scratch" in msg and f"needs {sms * per_sm} " in msg, msg
    finally:
        itr.red_set_knob(itr.RED_KNOB_FULL_CTAS_PER_SM, 0)
    x.fill_(0.5)
    assert _call_noalloc("sum", x, out) == itr.RED_OK
    assert abs(float(out[0]) - 0.5 * (1 << 28)) <= SUM_RTOL * 0.5 * (1 << 28)
