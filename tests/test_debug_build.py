"""The TA_DEBUG build of the library (device-side bounds checks on page-table lookups, TMA pool
rows and output rows) compiles for sm_103a and exports every function include/treeattn.h
declares (CPU)."""
import ctypes

from dag_packed_paged_gb300 import _native, build


def test_debug_library_builds_and_exports_every_declared_function():
    path = build.build(debug=True)
    assert path == build.LIB_DEBUG and path != build.LIB
    lib = ctypes.CDLL(path)
    for n in _native.header_functions():
        assert hasattr(lib, n), n


def test_bounds_error_code_is_declared():
    text = open(build.INCLUDE + "/treeattn.h").read()
    assert "#define TA_ERR_DEVICE_BOUNDS (-6)" in text
    assert _native.TA_ERR_DEVICE_BOUNDS == -6
