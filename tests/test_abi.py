"""The C-ABI library builds, loads without a GPU, exports every declared symbol,
and rejects invalid calls on the host (no device work is requested here)."""
import ctypes
import re
from pathlib import Path

import pytest

from volumetric_ultrasound_delay_gb300 import build as build_mod

HEADER = Path(__file__).resolve().parent.parent / "include" / "das.h"


@pytest.fixture(scope="module")
def libdas():
    build_mod.build()
    from volumetric_ultrasound_delay_gb300 import das
    return das.lib()


def declared_functions():
    text = re.sub(r"/\*.*?\*/", "", HEADER.read_text(), flags=re.S)
    return sorted(set(re.findall(r"\b(das_[a-z_0-9]+)\s*\(", text)))


def test_header_declares_the_boundary():
    names = declared_functions()
    for required in ("das_plan_create", "das_beamform", "das_plan_destroy", "das_permute"):
        assert required in names


def test_every_declared_symbol_is_exported(libdas):
    for name in declared_functions():
        assert hasattr(libdas, name), name


def test_binding_covers_every_symbol():
    from volumetric_ultrasound_delay_gb300 import das
    assert sorted(das._SIGS) == declared_functions()


def test_host_side_rejections(libdas):
    from volumetric_ultrasound_delay_gb300 import das
    h = ctypes.c_void_p()
    g = das._Grid(4, 4, 4, 0.0, 0.0, 0.01, 1e-3, 1e-3, 1e-3)
    rx = (ctypes.c_float * 3)(0.0, 0.0, 0.0)
    # null plan pointer, null grid, bad sizes, bad physics: all rejected before any CUDA call
    assert libdas.das_plan_create(None, ctypes.byref(g), rx, 1540.0, 20e6, 0.0, 1.5, 0, 1, 1, 1, 8) == das.DAS_ERR_INVALID_ARG
    assert libdas.das_plan_create(ctypes.byref(h), None, rx, 1540.0, 20e6, 0.0, 1.5, 0, 1, 1, 1, 8) == das.DAS_ERR_INVALID_ARG
    assert libdas.das_plan_create(ctypes.byref(h), ctypes.byref(g), rx, 1540.0, 20e6, 0.0, 1.5, 0, 0, 1, 1, 8) == das.DAS_ERR_INVALID_ARG
    assert libdas.das_plan_create(ctypes.byref(h), ctypes.byref(g), rx, -1.0, 20e6, 0.0, 1.5, 0, 1, 1, 1, 8) == das.DAS_ERR_INVALID_ARG
    assert libdas.das_plan_create(ctypes.byref(h), ctypes.byref(g), rx, 1540.0, 20e6, 0.0, 1.5, 7, 1, 1, 1, 8) == das.DAS_ERR_INVALID_ARG
    assert libdas.das_plan_create(ctypes.byref(h), ctypes.byref(g), rx, 1540.0, 20e6, 0.0, 1.5, 0, 1, 1, 1, 1 << 22) == das.DAS_ERR_INVALID_ARG
    assert h.value is None
    assert b"K must be" in libdas.das_last_error_string()
    bad = das._Grid(0, 4, 4, 0.0, 0.0, 0.01, 1e-3, 1e-3, 1e-3)
    assert libdas.das_plan_create(ctypes.byref(h), ctypes.byref(bad), rx, 1540.0, 20e6, 0.0, 1.5, 0, 1, 1, 1, 8) == das.DAS_ERR_INVALID_ARG
    # a grid carrying a voxel list goes through the list checks (a NaN position)
    pts = (ctypes.c_float * (3 * 64))(*([0.0] * (3 * 64 - 1) + [float("nan")]))
    listed = das._Grid(4, 4, 4, 0.0, 0.0, 0.01, 1e-3, 1e-3, 1e-3, ctypes.cast(pts, ctypes.c_void_p))
    assert libdas.das_plan_create(ctypes.byref(h), ctypes.byref(listed), rx, 1540.0, 20e6, 0.0, 1.5, 0, 1, 1, 1, 8) == das.DAS_ERR_INVALID_ARG
    assert b"voxel position" in libdas.das_last_error_string()
    # calls on a NULL plan
    assert libdas.das_beamform(None, None, None, None, None, None) == das.DAS_ERR_INVALID_ARG
    assert libdas.das_plan_set_option(None, 0, 0.0) == das.DAS_ERR_INVALID_ARG
    assert libdas.das_plan_launches(None, None) == das.DAS_ERR_INVALID_ARG
    assert libdas.das_beamform_host_volumes(None, 1, None, None, None, None, None) == das.DAS_ERR_INVALID_ARG
    # unknown dtypes; the half-precision records exist for plans and das_permute only
    assert libdas.das_plan_create(ctypes.byref(h), ctypes.byref(g), rx, 1540.0, 20e6, 0.0, 1.5, 6, 1, 1, 1, 8) == das.DAS_ERR_INVALID_ARG
    one = ctypes.create_string_buffer(1024)
    for dtype in (das.DAS_F16, das.DAS_C32H, 6):
        assert libdas.das_beamform_noalloc(ctypes.byref(g), one, 1540.0, 20e6, 0.0, 1.5, 0.0, dtype, 8, 1, 1, 8,
                                           one, one, one, one, None) == das.DAS_ERR_INVALID_ARG
        assert b"dtype" in libdas.das_last_error_string()
    assert libdas.das_plan_destroy(None) == das.DAS_OK
    # permute argument checks
    assert libdas.das_permute(None, None, 0, 1, 1, 1, 1, 0, 0, None) == das.DAS_ERR_INVALID_ARG
    buf = ctypes.create_string_buffer(64)
    assert libdas.das_permute(buf, buf, 0, 1, 1, 1, 4, 0, 0, None) == das.DAS_ERR_INVALID_ARG  # overlap
    assert libdas.das_permute(buf, ctypes.byref(buf, 32), 0, 1, 1, 1, 4, 4, 0, None) == das.DAS_ERR_INVALID_ARG  # bad layout
    assert libdas.das_permute(buf, ctypes.byref(buf, 32), 0, 1, 1, 1, 4, 0, 7, None) == das.DAS_ERR_INVALID_ARG  # bad storage
    assert libdas.das_permute(buf, ctypes.byref(buf, 32), 6, 1, 1, 1, 4, 0, 0, None) == das.DAS_ERR_INVALID_ARG  # bad dtype
    assert libdas.das_permute(buf, buf, das.DAS_F16, 1, 1, 1, 4, 0, 0, None) == das.DAS_ERR_INVALID_ARG  # overlap
    assert libdas.das_permute(buf, ctypes.byref(buf, 32), das.DAS_F16, 1, 1, 1, 4, 4, 0, None) == das.DAS_ERR_INVALID_ARG  # layout
    # element alignment: float32 needs 4 bytes, complex64 8, a half copy 2
    base = ctypes.addressof(buf) + (-ctypes.addressof(buf)) % 16
    big = ctypes.create_string_buffer(256)
    bbase = ctypes.addressof(big) + (-ctypes.addressof(big)) % 16
    assert libdas.das_permute(base + 2, bbase, 0, 1, 1, 1, 4, 0, 0, None) == das.DAS_ERR_INVALID_ARG
    assert b"aligned" in libdas.das_last_error_string()
    assert libdas.das_permute(base, bbase + 1, 0, 1, 1, 1, 4, 0, 0, None) == das.DAS_ERR_INVALID_ARG
    assert libdas.das_permute(base + 4, bbase, 1, 1, 1, 1, 2, 0, 0, None) == das.DAS_ERR_INVALID_ARG
    assert libdas.das_permute(base, bbase + 1, 0, 1, 1, 1, 4, 0, 1, None) == das.DAS_ERR_INVALID_ARG
    assert libdas.das_permute_bqmk_to_kqmb(base + 2, bbase, 0, 1, 1, 1, 4, None) == das.DAS_ERR_INVALID_ARG
    assert libdas.das_permute_bqmk_to_kqmb(None, None, 0, 1, 1, 1, 1, None) == das.DAS_ERR_INVALID_ARG
    assert libdas.das_permute_bqmk_to_kqmb(buf, buf, 0, 1, 1, 1, 4, None) == das.DAS_ERR_INVALID_ARG  # overlap
    assert libdas.das_permute_bqmk_to_kqmb(buf, ctypes.byref(buf, 32), 5, 1, 1, 1, 4, None) == das.DAS_ERR_INVALID_ARG
    assert libdas.das_version() == b"1.0.0"
