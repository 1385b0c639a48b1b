"""Seeded synthetic inputs for the five reduction workloads.

This module only draws random numbers and lays them out; it holds none of the
reductions' arithmetic, so the tests and the benchmark can feed the same
buffers to the CUDA path and to the CPU oracle.  Values come from
``torch.Generator(device).manual_seed(seed)``: the same seed gives the same
bits on the same device type (the CUDA and the CPU generator differ, which is
harmless because both sides of every comparison read one buffer).

Post-pass on every fp32 input:
  * exact zeros become +2**-10, so max / min never meet a +0/-0 tie;
  * values with 0 < |x| < FLT_MIN (denormals) also become +2**-10, so packed
    flush-to-zero arithmetic sees none (uniform draws are multiples of 2**-23
    and never hit this; it guards the normal draws);
  * no NaN or Inf can arise from these draws, and :func:`assert_finite` checks.

Workloads (sizes as stated by the benchmark's configuration list):
  1. full vector, N = 2**20, uniform[-1, 1), seed 0;
  2. dense rows 65536 x 1024 row-major, normal(0, 1), seed 1; the accum dst is
     uniform[-1, 1) from seed 101 (the workload gives no seed for it);
  3. full vector, N = 2**30 (4 GiB), normal(0, 1), seed 2;
  4. column products: fp32 4096 x 16384 uniform[0.999, 1.001], seed 3; int32
     64 x 65536 drawn uniformly from {-3, -2, -1, 1, 2, 3}, seed 4;
  5. ragged rows: 2**22 rows with lengths uniform on the integers 8..40
     inclusive, values uniform[-4, 4), int64 offsets, seed 5.
"""
from __future__ import annotations

import torch

TINY = 2.0 ** -10
FLT_MIN = 1.1754943508222875e-38

CFG1_N = 1 << 20
CFG2_ROWS, CFG2_LEN = 65536, 1024
CFG2_DST_SEED = 101
CFG3_N = 1 << 30
CFG4A_R, CFG4A_C = 4096, 16384
CFG4B_R, CFG4B_C = 64, 65536
CFG5_ROWS = 1 << 22
CFG5_MINLEN, CFG5_MAXLEN = 8, 40
INT_CHOICES = (-3, -2, -1, 1, 2, 3)


def _gen(seed: int, device) -> torch.Generator:
    g = torch.Generator(device=torch.device(device))
    g.manual_seed(int(seed))
    return g


def _post(x: torch.Tensor) -> torch.Tensor:
    """Replace exact zeros and denormals by +2**-10 (in place)."""
    bad = x.abs() < FLT_MIN
    x.masked_fill_(bad, TINY)
    return x


def uniform(shape, lo: float, hi: float, seed: int, device="cpu") -> torch.Tensor:
    """fp32 uniform[lo, hi) drawn as lo + (hi - lo) * rand, post-processed."""
    g = _gen(seed, device)
    x = torch.rand(shape, generator=g, device=device, dtype=torch.float32)
    x.mul_(hi - lo).add_(lo)
    return _post(x)


def normal(shape, seed: int, device="cpu") -> torch.Tensor:
    """fp32 standard normal draws, post-processed."""
    g = _gen(seed, device)
    x = torch.randn(shape, generator=g, device=device, dtype=torch.float32)
    return _post(x)


def int_choice(shape, choices, seed: int, device="cpu") -> torch.Tensor:
    """int32 values drawn uniformly from ``choices``."""
    g = _gen(seed, device)
    idx = torch.randint(0, len(choices), shape, generator=g, device=device)
    table = torch.tensor(choices, dtype=torch.int32, device=device)
    return table[idx]


def ragged_offsets(rows: int, minlen: int, maxlen: int, seed: int, device="cpu") -> torch.Tensor:
    """int64 offsets[rows + 1] of rows whose lengths are uniform on minlen..maxlen."""
    g = _gen(seed, device)
    lens = torch.randint(minlen, maxlen + 1, (rows,), generator=g, device=device, dtype=torch.int64)
    off = torch.zeros(rows + 1, dtype=torch.int64, device=device)
    torch.cumsum(lens, 0, out=off[1:])
    return off


def ragged_values(nnz: int, lo: float, hi: float, seed: int, device="cpu") -> torch.Tensor:
    """Packed fp32 values for ragged rows; drawn after the lengths (seed + 1000)."""
    return uniform((nnz,), lo, hi, seed + 1000, device)


def assert_finite(x: torch.Tensor) -> None:
    if x.is_floating_point() and not bool(torch.isfinite(x).all()):
        raise ValueError("synthetic input holds NaN or Inf")


# ------------------------------------------------------------ the workloads

def cfg1(device="cpu", n: int = CFG1_N):
    return uniform((n,), -1.0, 1.0, 0, device)


def cfg2(device="cpu", rows: int = CFG2_ROWS, length: int = CFG2_LEN):
    x = normal((rows, length), 1, device)
    dst = uniform((rows,), -1.0, 1.0, CFG2_DST_SEED, device)
    return x, dst


def cfg3(device="cpu", n: int = CFG3_N):
    return normal((n,), 2, device)


def cfg4a(device="cpu", R: int = CFG4A_R, C: int = CFG4A_C):
    return uniform((R, C), 0.999, 1.001, 3, device)


def cfg4b(device="cpu", R: int = CFG4B_R, C: int = CFG4B_C):
    return int_choice((R, C), INT_CHOICES, 4, device)


def cfg5(device="cpu", rows: int = CFG5_ROWS, minlen: int = CFG5_MINLEN, maxlen: int = CFG5_MAXLEN):
    off = ragged_offsets(rows, minlen, maxlen, 5, device)
    nnz = int(off[-1].item())
    x = ragged_values(nnz, -4.0, 4.0, 5, device)
    return x, off


# ------------------------------------------- column reductions, all types

COL_STORAGE = {"f32": torch.float32, "i32": torch.int32, "u32": torch.int32, "f16": torch.float16,
               "bf16": torch.bfloat16, "i16": torch.int16, "u16": torch.int16}


def col_input(op: str, dtype: str, shape, seed: int, device="cpu") -> torch.Tensor:
    """Seeded input for a column reduction of element type ``dtype`` ("f32",
    "i32", "u32", "f16", "bf16", "i16", "u16"); u16 / u32 come back in
    int16 / int32 storage holding the unsigned bit patterns.  Products get
    values that keep long products finite: uniform[0.99, 1.01] for floating
    types, {+-1, +-2, +-3} (unsigned: {1, 2, 3}) for integers; the other
    operators get uniform[-1, 1) floats or integers over the type's range."""
    g = _gen(seed, device)
    if dtype in ("f32", "f16", "bf16"):
        lo, hi = (0.99, 1.01) if op == "prod" else (-1.0, 1.0)
        x = torch.rand(shape, generator=g, device=device, dtype=torch.float32).mul_(hi - lo).add_(lo)
        return _post(x).to(COL_STORAGE[dtype])
    if op == "prod":
        choices = (1, 2, 3) if dtype in ("u16", "u32") else INT_CHOICES
        idx = torch.randint(0, len(choices), shape, generator=g, device=device)
        return torch.tensor(choices, dtype=torch.int64, device=device)[idx].to(COL_STORAGE[dtype])
    bits = 16 if dtype in ("i16", "u16") else 32
    # the type's full bit range, drawn in int64 and stored two's complement
    v = torch.randint(-(1 << (bits - 1)), 1 << (bits - 1), shape, generator=g, device=device, dtype=torch.int64)
    return v.to(COL_STORAGE[dtype])
