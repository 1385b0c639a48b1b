"""Pins of the CPU oracle to facts fixed outside the oracle itself.

Each check uses one of: the worked check a page gives (32-element sum), a
closed form, exact-arithmetic brute force on tiny inputs (``math.fsum``,
``fractions.Fraction``, Python big integers), or an invariant of the
definition.  They are chosen so that a dropped term, a wrong index or stride,
a wrong sign, a transposed operand or a mishandled remainder in the oracle
fails at least one of them.
"""
import math
from fractions import Fraction

import numpy as np
import pytest

import oracle
from conftest import golden_lines


def _grid_uniform(rng, n, lo=-1.0, hi=1.0):
    """fp32 values on the 2**-23 grid in [lo, hi), none exactly zero.

    Sums of up to 2**20 such values are exact in double, so the oracle's
    double sum must equal math.fsum bit for bit.
    """
    k = rng.integers(int(lo * 2**23), int(hi * 2**23), size=n)
    k[k == 0] = 1
    return (k.astype(np.float64) * 2.0**-23).astype(np.float32)


# ------------------------------------------------------------ page check

def test_sum32_page_demo():
    """Apache TVM docs, "reduction -> sm100_packed", "Demonstration program":
    B == sum(A) for a 32-element float32 vector (values A[i] = i)."""
    rows = dict((r[0], r[1:]) for r in golden_lines("sm100_packed_demo_sum32.txt"))
    n = int(rows["n"][0])
    a = np.array([float(v) for v in rows["A"]], np.float32)
    assert a.size == n == 32
    s, ab = oracle.full_sum(a)
    assert s == float(rows["B"][0]) == 496.0
    assert ab == 496.0


# ------------------------------------------------------------ full sum

@pytest.mark.parametrize("n", [1, 2, 7, 8, 9, 31, 32, 33, 1000, 4097, 1 << 20])
def test_sum_arange_closed_form(n):
    """sum_{i<n} i = n(n-1)/2, exact (all values and partial sums < 2**53)."""
    a = np.arange(n, dtype=np.float32)
    s, ab = oracle.full_sum(a)
    assert s == n * (n - 1) // 2
    assert ab == n * (n - 1) // 2


def test_sum_negated_arange():
    """Sign check: sum of -i is -n(n-1)/2 while sum |x| stays n(n-1)/2."""
    a = -np.arange(100, dtype=np.float32)
    s, ab = oracle.full_sum(a)
    assert s == -4950.0 and ab == 4950.0


def test_sum_bruteforce_fsum():
    """Every length 0..64 (covers chunk-of-8 remainders 0..7) against fsum."""
    rng = np.random.default_rng(11)
    for n in range(0, 65):
        for _ in range(3):
            a = _grid_uniform(rng, n, -4.0, 4.0)
            s, ab = oracle.full_sum(a)
            assert s == math.fsum(float(v) for v in a)
            assert ab == math.fsum(abs(float(v)) for v in a)


def test_sum_empty_is_zero():
    s, ab = oracle.full_sum(np.zeros(0, np.float32))
    assert s == 0.0 and ab == 0.0


def test_sum_accumulates_in_double():
    """2**24 + 1 + 1 + ... is lost in an fp32 accumulator but not in double."""
    a = np.ones(1001, np.float32)
    a[0] = 2.0**24
    s, _ = oracle.full_sum(a)
    assert s == 2.0**24 + 1000


# ------------------------------------------------------------ full max/min

def test_max_min_position_sweep():
    """The extreme is found at every index of every length 1..64."""
    rng = np.random.default_rng(12)
    for n in range(1, 65):
        base = _grid_uniform(rng, n, -1.0, 1.0)
        for p in range(n):
            a = base.copy()
            a[p] = 3.5
            assert oracle.full_max(a) == np.float32(3.5)
            a[p] = -3.5
            assert oracle.full_min(a) == np.float32(-3.5)


def test_max_min_bruteforce_and_duality():
    rng = np.random.default_rng(13)
    for n in (1, 5, 8, 13, 40, 257):
        a = _grid_uniform(rng, n, -2.0, 2.0)
        assert oracle.full_max(a) == max(a.tolist())
        assert oracle.full_min(a) == min(a.tolist())
        assert oracle.full_max(a) == -oracle.full_min(-a)


def test_max_min_empty_rejected():
    with pytest.raises(oracle.OracleError):
        oracle.full_max(np.zeros(0, np.float32))
    with pytest.raises(oracle.OracleError):
        oracle.full_min(np.zeros(0, np.float32))


# ------------------------------------------------------------ dense rows

@pytest.mark.parametrize("rows,length", [(1, 1), (3, 7), (5, 8), (4, 9), (7, 31), (6, 40), (2, 100)])
def test_rows_bruteforce(rows, length):
    rng = np.random.default_rng(rows * 100 + length)
    x = _grid_uniform(rng, rows * length, -4.0, 4.0).reshape(rows, length)
    s, ab = oracle.rows("sum", x, rows, length)
    mx = oracle.rows("max", x, rows, length)
    mn = oracle.rows("min", x, rows, length)
    for r in range(rows):
        row = [float(v) for v in x[r]]
        assert s[r] == math.fsum(row)
        assert ab[r] == math.fsum(abs(v) for v in row)
        assert mx[r] == max(row)
        assert mn[r] == min(row)


def test_rows_accum_closed_form():
    """Rows of ones: sum with accum = dst_old + len (exact); the old value is
    folded in once, not per element; max/min fold dst_old as one more value."""
    rows, length = 6, 37
    x = np.ones((rows, length), np.float32)
    dst = np.array([-0.5, 0.25, 100.0, -100.0, 1.5, 0.75], np.float32)
    s, ab = oracle.rows("sum", x, rows, length, accum=True, dst_old=dst)
    assert (s == dst.astype(np.float64) + length).all()
    assert (ab == np.abs(dst.astype(np.float64)) + length).all()
    mx = oracle.rows("max", x, rows, length, accum=True, dst_old=dst)
    mn = oracle.rows("min", x, rows, length, accum=True, dst_old=dst)
    assert mx.tolist() == [max(1.0, float(d)) for d in dst]
    assert mn.tolist() == [min(1.0, float(d)) for d in dst]


def test_rows_agree_with_full_per_row():
    """Stride check: row r of the matrix reduces like the slice x[r]."""
    rng = np.random.default_rng(14)
    rows, length = 9, 23
    x = _grid_uniform(rng, rows * length).reshape(rows, length)
    s, _ = oracle.rows("sum", x, rows, length)
    mx = oracle.rows("max", x, rows, length)
    for r in range(rows):
        assert s[r] == oracle.full_sum(x[r])[0]
        assert mx[r] == oracle.full_max(x[r])


def test_rows_len0():
    x = np.zeros((4, 0), np.float32)
    s, _ = oracle.rows("sum", x, 4, 0)
    assert (s == 0).all()
    dst = np.array([1.0, -2.0, 3.0, 0.5], np.float32)
    s, _ = oracle.rows("sum", x, 4, 0, accum=True, dst_old=dst)
    assert (s == dst).all()
    with pytest.raises(oracle.OracleError):
        oracle.rows("max", x, 4, 0)


# ------------------------------------------------------------ ragged rows

def test_ragged_matches_dense_layout():
    rng = np.random.default_rng(15)
    rows, length = 11, 19
    x = _grid_uniform(rng, rows * length)
    off = np.arange(rows + 1, dtype=np.int64) * length
    for op in ("max", "min"):
        assert (oracle.ragged(op, x, off) == oracle.rows(op, x, rows, length)).all()
    assert (oracle.ragged("sum", x, off)[0] == oracle.rows("sum", x, rows, length)[0]).all()


def test_ragged_bruteforce_with_empty_rows():
    """Lengths 0..40 (8..40 is the workload's range; 0 tests empty rows)."""
    rng = np.random.default_rng(16)
    lens = rng.integers(0, 41, size=200)
    lens[::17] = 0
    off = np.zeros(lens.size + 1, np.int64)
    off[1:] = np.cumsum(lens)
    x = _grid_uniform(rng, int(off[-1]), -4.0, 4.0)
    dst = _grid_uniform(rng, lens.size, -1.0, 1.0)
    for accum in (False, True):
        s, ab = oracle.ragged("sum", x, off, accum, dst)
        mx = oracle.ragged("max", x, off, accum, dst)
        mn = oracle.ragged("min", x, off, accum, dst)
        for r in range(lens.size):
            row = [float(v) for v in x[off[r]:off[r + 1]]]
            init = [float(dst[r])] if accum else []
            assert s[r] == math.fsum(init + row)
            assert ab[r] == math.fsum(abs(v) for v in init + row)
            assert mx[r] == max(init + row, default=-math.inf)
            assert mn[r] == min(init + row, default=math.inf)


def test_ragged_rejects_decreasing_offsets():
    x = np.ones(10, np.float32)
    with pytest.raises(oracle.OracleError):
        oracle.ragged("sum", x, np.array([0, 5, 3, 10], np.int64))
    with pytest.raises(oracle.OracleError):
        oracle.ragged("max", x, np.array([1, 5, 10], np.int64))


# ------------------------------------------------------------ TCOLPROD f32

def _f32_of(fr: Fraction) -> np.float32:
    """Nearest float32 of an exact rational whose numerator and denominator
    fit in 53 bits (so Fraction -> double is exact, then one rounding)."""
    return np.float32(fr.numerator / fr.denominator)


def test_tcolprod_16x16_page_example():
    """pto-isa docs, "TCOLPROD", "Examples": 16 x 16 float tile -> 1 x 16,
    with constant columns whose products have closed forms."""
    lines = golden_lines("tcolprod_16x16.txt")
    R = int(lines[0][1]); C = int(lines[1][1])
    cs, exp = [], []
    for j, c, frac in lines[2:]:
        cs.append(np.float32(float(c)))
        exp.append(Fraction(frac))
    x = np.tile(np.array(cs, np.float32), (R, 1))
    out, outd = oracle.colprod_f32(x, R, C, want_double=True)
    for j in range(C):
        assert out[j] == _f32_of(exp[j]), j
        assert outd[j] == exp[j].numerator / exp[j].denominator, j


@pytest.mark.parametrize("c,R", [(1.0, 100), (-1.0, 99), (-1.0, 100), (2.0, 100), (0.5, 120), (-2.0, 37)])
def test_colprod_constant_columns(c, R):
    C = 7
    x = np.full((R, C), c, np.float32)
    out = oracle.colprod_f32(x, R, C)
    assert (out == np.float32(c ** R)).all()


def test_colprod_not_transposed():
    """x[i,j] = c_j * s_i with s_i = +-1: out[j] = c_j**R * prod(s); a product
    taken along rows instead of columns gives a different answer."""
    R, C = 5, 3
    c = np.array([2.0, 0.5, -3.0], np.float32)
    s = np.array([1, -1, -1, -1, 1], np.float32)
    x = (s[:, None] * c[None, :]).astype(np.float32)
    out = oracle.colprod_f32(x, R, C)
    assert out.tolist() == [float(cj) ** R * -1.0 for cj in c]


def test_colprod_bruteforce_exact():
    rng = np.random.default_rng(17)
    for R, C in [(1, 1), (1, 5), (3, 4), (8, 3), (13, 6), (40, 2)]:
        x = rng.uniform(0.5, 1.5, size=(R, C)).astype(np.float32)
        out, outd = oracle.colprod_f32(x, R, C, want_double=True)
        for j in range(C):
            ex = math.prod(Fraction(float(v)) for v in x[:, j])
            rel = abs(Fraction(float(outd[j])) - ex) / ex
            assert rel <= R * 2.0**-53
            # one fp32 rounding of a value within R ulp(double) of exact
            ref = np.float32(float(ex))
            assert abs(int(out[j].view(np.int32)) - int(ref.view(np.int32))) <= 1


def test_colprod_early_return_leaves_dst():
    """pto-isa docs, "TCOLPROD", "Constraints": R == 0 or C == 0 returns early."""
    sentinel = np.full(4, 7.25, np.float32)
    oracle.colprod_f32(np.zeros((0, 4), np.float32), 0, 4, out_f=sentinel)
    assert (sentinel == 7.25).all()
    oracle.colprod_f32(np.zeros((3, 0), np.float32), 3, 0, out_f=sentinel)
    assert (sentinel == 7.25).all()
    isent = np.full(4, -9, np.int32)
    oracle.colprod_i32(np.zeros((0, 4), np.int32), 0, 4, out=isent)
    assert (isent == -9).all()


# ------------------------------------------------------------ TCOLPROD i32

def test_colprod_i32_wrap_closed_forms():
    for c, R, expected in golden_lines("tcolprod_i32_wrap.txt"):
        c, R, expected = int(c), int(R), int(expected)
        x = np.full((R, 3), c, np.int32)
        out = oracle.colprod_i32(x, R, 3)
        assert (out == expected).all(), (c, R)


def _wrap32(v: int) -> int:
    v %= 1 << 32
    return v - (1 << 32) if v >= 1 << 31 else v


def test_colprod_i32_bruteforce_bigint():
    rng = np.random.default_rng(18)
    for R, C in [(1, 4), (7, 5), (33, 3), (64, 9), (100, 2)]:
        x = rng.choice(np.array([-3, -2, -1, 1, 2, 3], np.int32), size=(R, C))
        out = oracle.colprod_i32(x, R, C)
        for j in range(C):
            assert out[j] == _wrap32(math.prod(int(v) for v in x[:, j]))


def test_colprod_i32_large_values_wrap():
    rng = np.random.default_rng(19)
    R, C = 9, 6
    x = rng.integers(-2**31, 2**31, size=(R, C), dtype=np.int64).astype(np.int32)
    out = oracle.colprod_i32(x, R, C)
    for j in range(C):
        assert out[j] == _wrap32(math.prod(int(v) for v in x[:, j]))


# ------------------------------------------------ thread-scope fold order

def _fold_cases():
    for name, accum, dst, expected, *vals in golden_lines("sm100_packed_fold_order.txt"):
        yield name, bool(int(accum)), float(dst), float(expected), np.array([float(v) for v in vals], np.float32)


def test_thread_sum_hand_worked_rounding_order():
    """Apache TVM docs, "reduction -> sm100_packed", "Algorithm": the page's
    fold order, worked by hand in fp32 (tests/golden/sm100_packed_fold_order.txt)."""
    for name, accum, dst, expected, a in _fold_cases():
        assert oracle.thread_sum(a, accum, dst) == np.float32(expected), name


def test_thread_sum_page_demo():
    """"Demonstration program": B == sum(A) for 32 float32 values."""
    assert oracle.thread_sum(np.arange(32, dtype=np.float32)) == np.float32(496)


@pytest.mark.parametrize("n", list(range(1, 65)))
def test_thread_sum_exact_when_no_rounding(n):
    """Integer values with small sums are exact in every order: closed form."""
    a = np.arange(1, n + 1, dtype=np.float32)
    assert oracle.thread_sum(a) == np.float32(n * (n + 1) // 2)
    assert oracle.thread_sum(a, True, 7.0) == np.float32(n * (n + 1) // 2 + 7)


def test_thread_sum_within_the_fp32_error_bound():
    """Random data: |fold - exact| <= (n - 1) * 2**-24 * sum|a| (any fp32
    summation order of n terms satisfies this)."""
    rng = np.random.default_rng(31)
    for n in range(1, 65):
        a = _grid_uniform(rng, n, -4.0, 4.0)
        exact = math.fsum(float(v) for v in a)
        bound = max(n - 1, 1) * 2.0**-24 * math.fsum(abs(float(v)) for v in a)
        assert abs(float(oracle.thread_sum(a)) - exact) <= bound, n


# ------------------------------------------------ column reductions, all types

def test_half_decode_exhaustive():
    """Every binary16 bit pattern decodes as numpy's float16 does."""
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    ref = bits.view(np.float16).astype(np.float64)
    got = np.array([oracle.half_to_double(int(b)) for b in bits])
    same = (got == ref) | (np.isnan(got) & np.isnan(ref))
    assert same.all()


def test_bf16_decode_exhaustive():
    """Every bfloat16 bit pattern decodes as torch's bfloat16 does."""
    import torch
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    ref = torch.from_numpy(bits.view(np.int16).copy()).view(torch.bfloat16).to(torch.float64).numpy()
    got = np.array([oracle.bf16_to_double(int(b)) for b in bits])
    same = (got == ref) | (np.isnan(got) & np.isnan(ref))
    assert same.all()


def _wrap(v, bits, signed):
    v %= 1 << bits
    return v - (1 << bits) if signed and v >= 1 << (bits - 1) else v


@pytest.mark.parametrize("dtype,bits,signed", [("i32", 32, True), ("u32", 32, False), ("i16", 16, True),
                                               ("u16", 16, False)])
def test_int_cols_bruteforce(dtype, bits, signed):
    rng = np.random.default_rng(bits + signed)
    npt = {"i32": np.int32, "u32": np.uint32, "i16": np.int16, "u16": np.uint16}[dtype]
    info = np.iinfo(npt)
    for R, C in [(1, 3), (5, 4), (17, 6), (64, 3)]:
        x = rng.integers(int(info.min), int(info.max) + 1, size=(R, C), dtype=np.int64).astype(npt)
        for op in ("sum", "prod", "max", "min"):
            got = oracle.cols(op, dtype, x, R, C)
            for j in range(C):
                col = [int(v) for v in x[:, j]]
                if op == "sum":
                    ref = _wrap(sum(col), bits, signed)
                elif op == "prod":
                    ref = _wrap(math.prod(col), bits, signed)
                else:
                    ref = max(col) if op == "max" else min(col)
                assert got[j] == ref, (dtype, op, R, C, j)


def test_int16_wrap_closed_forms():
    """2^15 wraps to -32768 in int16 and 2^16 to 0; 3^11 = 177147 wraps to
    177147 - 3 * 65536 = -19461; the unsigned types wrap to the residue."""
    for c, R, dtype, ref in [(2, 15, "i16", -32768), (2, 16, "i16", 0), (3, 11, "i16", 177147 - 3 * 65536),
                             (3, 11, "u16", 177147 % 65536), (2, 32, "u32", 0), (3, 21, "u32", 3**21 % 2**32),
                             (-1, 7, "i16", -1)]:
        npt = {"i16": np.int16, "u16": np.uint16, "u32": np.uint32}[dtype]
        x = np.full((R, 2), c, np.int64).astype(npt)
        assert (oracle.cols("prod", dtype, x, R, 2) == ref).all(), (c, R, dtype)


@pytest.mark.parametrize("dtype", ["f32", "f16", "bf16"])
def test_float_cols_bruteforce(dtype):
    import torch
    rng = np.random.default_rng(5)
    for R, C in [(1, 2), (3, 5), (16, 16), (40, 3)]:
        v = rng.uniform(0.5, 1.5, size=(R, C)).astype(np.float32)
        if dtype == "f32":
            x = v
            vals = v.astype(np.float64)
        elif dtype == "f16":
            x = v.astype(np.float16)
            vals = x.astype(np.float64)
        else:
            t = torch.from_numpy(v).to(torch.bfloat16)
            x = t.view(torch.int16).numpy()
            vals = t.to(torch.float64).numpy()
        for op in ("sum", "prod", "max", "min"):
            got, ab = oracle.cols(op, dtype, x, R, C)
            for j in range(C):
                col = [float(a) for a in vals[:, j]]
                assert ab[j] == math.fsum(abs(a) for a in col)
                if op == "sum":
                    assert got[j] == math.fsum(col)           # exact: few short values
                elif op == "prod":
                    ex = math.prod(Fraction(a) for a in col)
                    assert abs(Fraction(got[j]) - ex) <= abs(ex) * R * Fraction(2) ** -53
                else:
                    assert got[j] == (max(col) if op == "max" else min(col))


def test_cols_not_transposed_and_early_return():
    x = np.array([[1, 2, 3], [4, 5, 6]], np.int32)
    assert oracle.cols("sum", "i32", x, 2, 3).tolist() == [5, 7, 9]
    assert oracle.cols("prod", "i32", x, 2, 3).tolist() == [4, 10, 18]
    sentinel = np.full(3, 7, np.int64)
    oracle.cols("sum", "i32", np.zeros((0, 3), np.int32), 0, 3, out=sentinel)
    assert sentinel.tolist() == [7, 7, 7]
    fs = np.full(3, 2.5)
    oracle.cols("max", "f16", np.zeros((0, 3), np.float16), 0, 3, out=fs)
    assert fs.tolist() == [2.5, 2.5, 2.5]


def test_cols_f32_product_matches_colprod():
    rng = np.random.default_rng(6)
    x = rng.uniform(0.9, 1.1, size=(30, 7)).astype(np.float32)
    got, _ = oracle.cols("prod", "f32", x, 30, 7)
    _, pd = oracle.colprod_f32(x, 30, 7, want_double=True)
    assert (got == pd).all()


# ------------------------------------------------ typed rows (all element types)

def test_rows_typed_agree_with_columns_of_the_transpose():
    """Row r of x is column r of x^T: the typed row oracle and the column
    oracle (pinned above) must agree on every type and operator."""
    rng = np.random.default_rng(8)
    for dtype, npt in [("i32", np.int32), ("u32", np.uint32), ("i16", np.int16), ("u16", np.uint16)]:
        info = np.iinfo(npt)
        x = rng.integers(int(info.min), int(info.max) + 1, size=(6, 11), dtype=np.int64).astype(npt)
        for op in ("sum", "prod", "max", "min"):
            assert (oracle.rows_typed(op, dtype, x, 6, 11) ==
                    oracle.cols(op, dtype, np.ascontiguousarray(x.T), 11, 6)).all(), (dtype, op)
    x = rng.uniform(0.5, 1.5, size=(5, 9)).astype(np.float16)
    for op in ("sum", "prod", "max", "min"):
        a, _ = oracle.rows_typed(op, "f16", x, 5, 9)
        b, _ = oracle.cols(op, "f16", np.ascontiguousarray(x.T), 9, 5)
        assert (a == b).all(), op


def test_rows_typed_accum_and_empty():
    x = np.array([[2, 3], [4, 5]], np.int16)
    old = np.array([10, -1], np.int16)
    assert oracle.rows_typed("sum", "i16", x, 2, 2, True, old).tolist() == [15, 8]
    assert oracle.rows_typed("prod", "i16", x, 2, 2, True, old).tolist() == [60, -20]
    assert oracle.rows_typed("max", "i16", x, 2, 2, True, old).tolist() == [10, 5]
    e = np.zeros((3, 0), np.int32)
    assert oracle.rows_typed("prod", "i32", e, 3, 0).tolist() == [1, 1, 1]
    assert oracle.rows_typed("sum", "i32", e, 3, 0).tolist() == [0, 0, 0]
    with pytest.raises(oracle.OracleError):
        oracle.rows_typed("max", "i32", e, 3, 0)
    # the empty product is 1 and the empty sum 0 for floating types too
    for dt, npt in (("f32", np.float32), ("f16", np.float16)):
        ef = np.zeros((3, 0), npt)
        assert oracle.rows_typed("prod", dt, ef, 3, 0)[0].tolist() == [1.0, 1.0, 1.0]
        assert oracle.rows_typed("sum", dt, ef, 3, 0)[0].tolist() == [0.0, 0.0, 0.0]
    r, _ = oracle.rows_typed("sum", "f16", np.full((1, 4), 0.5, np.float16), 1, 4, True,
                             np.array([1.0], np.float16))
    assert r.tolist() == [3.0]
