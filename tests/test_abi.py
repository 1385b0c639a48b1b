"""The C ABI library loads, exports every function include/red.h declares, and
rejects bad arguments on the host before touching the GPU (no compute call)."""
import ctypes
import os
import re

import pytest

from conftest import ROOT

HEADER = os.path.join(ROOT, "include", "red.h")


@pytest.fixture(scope="module")
def lib():
    from int_tensor_reductions_gb300 import _build, _binding
    _build.build_lib()
    return _binding.lib()


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    names = re.findall(r"^\s*(?:const\s+)?\w+\s*\*?\s*(red_\w+)\s*\(", text, flags=re.M)
    return sorted(set(names))


def test_header_declares_the_entry_points():
    names = declared_functions()
    for n in ("red_full", "red_rows", "red_rows_ragged", "red_colprod", "red_set_full_mode",
              "red_last_error", "red_release_workspace", "red_version"):
        assert n in names


def test_every_declared_symbol_is_exported(lib):
    missing = [n for n in declared_functions() if not hasattr(lib, n)]
    assert not missing, missing


def test_version(lib):
    assert lib.red_version() == 2


def _err(lib):
    return lib.red_last_error().decode()


def test_full_rejects_bad_arguments(lib):
    from int_tensor_reductions_gb300 import RED_EINVAL, RED_SUM, RED_MAX
    assert lib.red_full(7, 0x1000, 8, 0x2000, None) == RED_EINVAL
    assert "unknown op" in _err(lib)
    assert lib.red_full(RED_SUM, 0x1000, -1, 0x2000, None) == RED_EINVAL
    assert lib.red_full(RED_SUM, None, 8, 0x2000, None) == RED_EINVAL
    assert lib.red_full(RED_SUM, 0x1000, 8, None, None) == RED_EINVAL
    assert lib.red_full(RED_SUM, 0x1001, 8, 0x2000, None) == RED_EINVAL  # misaligned x
    assert lib.red_full(RED_MAX, None, 0, 0x2000, None) == RED_EINVAL    # max of nothing
    assert "empty" in _err(lib)


def test_rows_reject_bad_arguments(lib):
    from int_tensor_reductions_gb300 import RED_EINVAL, RED_OK, RED_SUM, RED_MIN
    assert lib.red_rows(RED_SUM, 0x1000, -2, 4, 0, 0x2000, None) == RED_EINVAL
    assert lib.red_rows(RED_SUM, 0x1000, 2, -4, 0, 0x2000, None) == RED_EINVAL
    assert lib.red_rows(RED_SUM, 0x1000, 1 << 40, 1 << 40, 0, 0x2000, None) == RED_EINVAL
    assert lib.red_rows(RED_MIN, 0x1000, 3, 0, 0, 0x2000, None) == RED_EINVAL
    assert lib.red_rows(RED_SUM, 0x1000, 0, 5, 0, None, None) == RED_OK   # nothing to do
    assert lib.red_rows(RED_SUM, 0x1000, 3, 0, 1, 0x2000, None) == RED_OK  # accum, empty rows
    assert lib.red_rows_ragged(RED_SUM, 0x1000, 0x3004, 4, 10, 0, 0x2000, None) == RED_EINVAL
    assert lib.red_rows_ragged(RED_SUM, 0x1000, None, 4, 10, 0, 0x2000, None) == RED_EINVAL
    assert lib.red_rows_ragged(9, 0x1000, 0x3000, 4, 10, 0, 0x2000, None) == RED_EINVAL


def test_colprod_rejects_and_returns_early(lib):
    from int_tensor_reductions_gb300 import RED_EINVAL, RED_F32, RED_OK
    assert lib.red_colprod(9, 0x1000, 4, 4, 0x2000, None) == RED_EINVAL
    assert lib.red_cols(4, RED_F32, 0x1000, 4, 4, 0x2000, None) == RED_EINVAL   # unknown op
    assert lib.red_cols(3, 7, 0x1000, 4, 4, 0x2000, None) == RED_EINVAL         # unknown dtype
    assert lib.red_cols(0, RED_F32, 0x1002, 4, 4, 0x2000, None) == RED_EINVAL   # f32 at 2-byte offset
    assert lib.red_cols(0, 2, 0x1001, 4, 4, 0x2000, None) == RED_EINVAL         # f16 at odd address
    assert lib.red_cols(1, 4, None, 0, 4, None, None) == RED_OK                 # early return
    assert lib.red_colprod(RED_F32, 0x1000, -1, 4, 0x2000, None) == RED_EINVAL
    # pto-isa docs, "TCOLPROD", "Constraints": empty tile -> early return
    assert lib.red_colprod(RED_F32, None, 0, 4, None, None) == RED_OK
    assert lib.red_colprod(RED_F32, None, 4, 0, None, None) == RED_OK


def test_cols_ld_rejects_and_returns_early(lib):
    """Row stride of the valid region (pto-isa docs, "TCOLPROD", "Math
    Interpretation": R x C = ValidRow x ValidCol of a wider row-major tile)."""
    from int_tensor_reductions_gb300 import RED_EINVAL, RED_F32, RED_OK
    assert lib.red_cols_ld(0, RED_F32, 0x1000, 4, 8, 7, 0x2000, None) == RED_EINVAL   # ld < C
    assert lib.red_cols_ld(0, RED_F32, 0x1000, 1 << 40, 8, 1 << 20, 0x2000, None) == RED_EINVAL  # R * ld too big
    assert lib.red_cols_ld(3, RED_F32, None, 0, 8, 16, None, None) == RED_OK          # empty: early return
    assert lib.red_cols_ld(3, RED_F32, None, 4, 0, 16, None, None) == RED_OK


def test_element_count_limit_is_2_pow_44(lib):
    """Every element count is at most 2^44 (include/red.h, "Sizes"); one
    more is refused on the host, before any CUDA call."""
    from int_tensor_reductions_gb300 import RED_EINVAL, RED_F32, RED_SUM
    big = (1 << 44) + 1
    assert lib.red_full(RED_SUM, 0x1000, big, 0x2000, None) == RED_EINVAL
    assert "out of range" in _err(lib)
    assert lib.red_full_noalloc(RED_SUM, 0x1000, big, 0x2000, None) == RED_EINVAL
    assert lib.red_full_stats(0x1000, big, 0x2000, None) == RED_EINVAL
    assert lib.red_full_typed(RED_SUM, RED_F32, 0x1000, big, 0x2000, None) == RED_EINVAL
    assert lib.red_rows(RED_SUM, 0x1000, 1, big, 0, 0x2000, None) == RED_EINVAL
    assert lib.red_rows(RED_SUM, 0x1000, (1 << 22) + 1, 1 << 22, 0, 0x2000, None) == RED_EINVAL
    assert lib.red_rows_typed(RED_SUM, RED_F32, 0x1000, big, 1, 0, 0x2000, None) == RED_EINVAL
    assert lib.red_rows_ragged(RED_SUM, 0x1000, 0x3000, 4, big, 0, 0x2000, None) == RED_EINVAL
    assert lib.red_cols(RED_SUM, RED_F32, 0x1000, (1 << 30) + 1, 1 << 14, 0x2000, None) == RED_EINVAL


def test_knobs_and_modes(lib):
    import int_tensor_reductions_gb300 as itr
    assert lib.red_set_full_mode(9) == itr.RED_EINVAL
    for m in (itr.RED_MODE_TWO_PASS, itr.RED_MODE_LAST_BLOCK, itr.RED_MODE_ATOMIC):
        itr.red_set_full_mode(m)
        assert itr.red_get_full_mode() == m
    itr.red_set_full_mode(itr.RED_MODE_AUTO)
    assert itr.red_get_full_mode() == itr.RED_MODE_AUTO
    assert lib.red_set_knob(itr.RED_KNOB_ROWS_GROUP, 3) == itr.RED_EINVAL
    itr.red_set_knob(itr.RED_KNOB_ROWS_GROUP, 8)
    assert itr.red_get_knob(itr.RED_KNOB_ROWS_GROUP) == 8
    itr.red_set_knob(itr.RED_KNOB_ROWS_GROUP, 0)
    assert lib.red_set_knob(itr.RED_KNOB_RAGGED_STAGED, 3) == itr.RED_EINVAL
    for v in (1, 2, 0):
        itr.red_set_knob(itr.RED_KNOB_RAGGED_STAGED, v)
        assert itr.red_get_knob(itr.RED_KNOB_RAGGED_STAGED) == v
    assert lib.red_get_knob(99) == itr.RED_EINVAL


def test_binding_refuses_cpu_tensors():
    import torch
    import int_tensor_reductions_gb300 as itr
    with pytest.raises(ValueError):
        itr.red_full("sum", torch.ones(8))


def test_c_client_compiles_and_links(lib, tmp_path):
    """tests/c/red_c_client.c (run on the GPU by test_gpu_c_client.py) builds
    against red.h as C99 and links against libred.so and the CUDA runtime."""
    import subprocess
    cuda = os.environ.get("CUDA_HOME", "/usr/local/cuda")
    pkg = os.path.dirname(lib._name)
    subprocess.run(["gcc", "-std=c99", "-O2", "-Wall", "-Wextra", "-Werror", "-I" + os.path.join(ROOT, "include"),
                    "-I" + os.path.join(cuda, "include"), os.path.join(ROOT, "tests", "c", "red_c_client.c"),
                    "-o", str(tmp_path / "client"), "-L" + pkg, "-lred", "-L" + os.path.join(cuda, "lib64"),
                    "-lcudart"], check=True)
