"""The library's calls captured into a CUDA graph (after a first eager call
has created the device's workspace) and replayed: same results as eager
calls, also after the inputs change in place between replays."""
import numpy as np
import pytest
import torch

import int_tensor_reductions_gb300 as itr
from int_tensor_reductions_gb300 import synth
from gpu_util import lib_ready, to_host

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    lib_ready()


def test_capture_and_replay_matches_eager():
    dev = torch.device("cuda")
    x = synth.normal((3_000_001,), 1, device=dev)
    m = synth.normal((4096, 1000), 2, device=dev)
    v, off = synth.cfg5(device=dev, rows=20000)
    c = synth.uniform((1024, 4096), 0.99, 1.01, 3, device=dev)
    h = synth.col_input("sum", "f16", (512, 2048), 4, device=dev)
    outs = {k: torch.empty(n, device=dev) for k, n in
            (("full", 1), ("stats", 4), ("rows", 4096), ("ragged", 20000), ("colprod", 4096))}
    oh = torch.empty(2048, dtype=torch.float16, device=dev)

    def calls():
        itr.red_full("sum", x, outs["full"])
        itr.red_full_stats(x, outs["stats"])
        itr.red_rows("max", m, out=outs["rows"])
        itr.red_rows_ragged("min", v, off, out=outs["ragged"])
        itr.red_colprod(c, outs["colprod"])
        itr.red_cols("sum", h, oh)

    def snapshot():
        torch.cuda.synchronize()
        return {k: to_host(t).copy() for k, t in outs.items()} | {"f16": to_host(oh).copy()}

    calls()  # eager: creates the workspace, caches the launch shapes
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        calls()
    for trial in range(2):
        for t, seed in ((x, 10), (m, 11), (v, 12), (c, 13)):
            t.copy_(synth.uniform(t.shape, 0.99, 1.01, seed + trial, device=dev) if t is c
                    else synth.normal(t.shape, seed + trial, device=dev))
        h.copy_(synth.col_input("sum", "f16", h.shape, 14 + trial, device=dev))
        g.replay()
        replayed = snapshot()
        calls()
        eager = snapshot()
        for k in eager:
            # the same kernels in the same launch shapes: bit for bit
            assert np.array_equal(replayed[k].view(np.uint8), eager[k].view(np.uint8)), (trial, k)
