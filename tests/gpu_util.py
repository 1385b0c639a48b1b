"""Helpers of the GPU parity tests: tolerances and comparisons against the
oracle.

Tolerances (stated by the workload definition and used everywhere):
  * fp32 sums: |gpu - exact| <= 1e-5 * sum|x| (plus |old dst| with accum);
  * max / min: bit-exact (inputs hold no NaN and no +-0 ties);
  * fp32 column products: |gpu - p| <= 5e-4 * |p|, p the double product;
  * int32 column products: bit-exact (wrapping modulo 2**32).
"""
import numpy as np
import torch

SUM_RTOL = 1e-5
PROD_RTOL = 5e-4


def lib_ready():
    from int_tensor_reductions_gb300 import _build
    _build.build_lib()


def to_host(t: torch.Tensor) -> np.ndarray:
    return t.detach().cpu().numpy()


def check_sum(gpu, exact, abs_sum, what=""):
    gpu = np.asarray(gpu, np.float64).reshape(-1)
    exact = np.asarray(exact, np.float64).reshape(-1)
    bound = SUM_RTOL * np.asarray(abs_sum, np.float64).reshape(-1)
    err = np.abs(gpu - exact)
    bad = np.nonzero(~(err <= bound))[0]
    assert bad.size == 0, (f"{what}: {bad.size} sums out of tolerance, first at {bad[0]}: "
                           f"gpu {gpu[bad[0]]!r} exact {exact[bad[0]]!r} bound {bound[bad[0]]!r}")


def check_exact(gpu, ref, what=""):
    gpu = np.asarray(gpu).reshape(-1)
    ref = np.asarray(ref).reshape(-1)
    assert gpu.dtype == ref.dtype, (gpu.dtype, ref.dtype)
    neq = np.nonzero(gpu.view(np.uint32) != ref.view(np.uint32))[0] if gpu.dtype.itemsize == 4 else \
        np.nonzero(gpu != ref)[0]
    assert neq.size == 0, (f"{what}: {neq.size} mismatches, first at {neq[0]}: "
                           f"gpu {gpu[neq[0]]!r} ref {ref[neq[0]]!r}")


def check_prod(gpu, exact_d, what=""):
    gpu = np.asarray(gpu, np.float64).reshape(-1)
    exact_d = np.asarray(exact_d, np.float64).reshape(-1)
    err = np.abs(gpu - exact_d)
    bound = PROD_RTOL * np.abs(exact_d)
    bad = np.nonzero(~(err <= bound))[0]
    assert bad.size == 0, (f"{what}: {bad.size} products out of tolerance, first at {bad[0]}: "
                           f"gpu {gpu[bad[0]]!r} exact {exact_d[bad[0]]!r}")
