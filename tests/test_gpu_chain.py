"""Library calls that consume the previous call's output, queued back to back
on one stream with no host synchronisation between them.

Every kernel is launched with programmatic dependent launch, so the next
kernel may already be resident while the previous one drains; each kernel
waits for its predecessors before touching memory.  Integer-valued fp32
inputs keep every sum exact, so a kernel that read a predecessor's output
too early would show up as a wrong value, not as rounding."""
import numpy as np
import pytest
import torch

import int_tensor_reductions_gb300 as itr
from gpu_util import lib_ready, to_host

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    lib_ready()


def _int_valued(shape, seed):
    g = torch.Generator(device="cuda")
    g.manual_seed(seed)
    return torch.randint(-3, 4, shape, generator=g, device="cuda").to(torch.float32)


def test_rows_accum_chain():
    """out += row sums, ten times; then a max and a min row pass folded into
    the same buffer (each call reads what the one before wrote)."""
    rows, length = 4096, 1000
    x = _int_valued((rows, length), 1)
    out = torch.zeros(rows, device="cuda")
    for _ in range(10):
        itr.red_rows("sum", x, accum=True, out=out)
    xh = to_host(x).astype(np.float64)
    want = 10 * xh.sum(axis=1)
    assert np.array_equal(to_host(out).astype(np.float64), want)
    itr.red_rows("max", x, accum=True, out=out)
    itr.red_rows("min", x, accum=True, out=out)
    want = np.minimum(np.maximum(want, xh.max(axis=1)), xh.min(axis=1))
    assert np.array_equal(to_host(out).astype(np.float64), want)


def test_cols_then_full_chain():
    """Column sums of a matrix, then the full sum and max of that result, then
    the ragged row sums of it (offsets cut the column sums into rows)."""
    R, C = 512, 8192
    x = _int_valued((R, C), 2)
    cs = torch.empty(C, device="cuda")
    tot = torch.empty(1, device="cuda")
    mx = torch.empty(1, device="cuda")
    off = torch.arange(0, C + 1, 64, dtype=torch.int64, device="cuda")
    rr = torch.empty(off.numel() - 1, device="cuda")
    for _ in range(5):
        itr.red_cols("sum", x, cs)
        itr.red_full("sum", cs, tot)
        itr.red_full("max", cs, mx)
        itr.red_rows_ragged("sum", cs, off, out=rr)
    colsum = to_host(x).astype(np.float64).sum(axis=0)
    assert np.array_equal(to_host(cs).astype(np.float64), colsum)
    assert float(to_host(tot)[0]) == colsum.sum()
    assert float(to_host(mx)[0]) == colsum.max()
    assert np.array_equal(to_host(rr).astype(np.float64), colsum.reshape(-1, 64).sum(axis=1))


def test_stats_and_typed_chain():
    """Fused row statistics feed a typed full reduction and a thread-scope
    row pass over the (rows x 4) statistics matrix."""
    rows, length = 2048, 512
    x = _int_valued((rows, length), 3)
    st = torch.empty((rows, 4), device="cuda")
    s_all = torch.empty(1, device="cuda")
    per_stat = torch.empty(rows, device="cuda")
    for _ in range(5):
        itr.red_rows_stats(x, st)
        itr.red_full_typed("sum", st.view(-1), s_all)
        itr.red_rows_thread("sum", st, out=per_stat)
    xh = to_host(x).astype(np.float64)
    want = np.stack([xh.sum(1), xh.max(1), xh.min(1), np.abs(xh).sum(1)], axis=1)
    assert np.array_equal(to_host(st).astype(np.float64), want)
    assert float(to_host(s_all)[0]) == want.sum()
    assert np.array_equal(to_host(per_stat).astype(np.float64), want.sum(axis=1))
