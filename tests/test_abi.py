"""The C ABI library loads and exports every function include/treeattn.h declares (CPU)."""
import ctypes

from dag_packed_paged_gb300 import _native, build


def test_library_exports_every_declared_function():
    build.build()
    lib = _native.lib()
    names = _native.header_functions()
    assert {"tree_attn_plan", "tree_attn_fwd", "tree_attn_bwd"} <= set(names)
    for n in names:
        assert hasattr(lib, n), n


def test_struct_layouts_match_header():
    assert ctypes.sizeof(_native.ta_branch) == 24
    assert ctypes.sizeof(_native.ta_mount) == 20
    assert ctypes.sizeof(_native.ta_config) == 32
    from dag_packed_paged_gb300 import workloads as W
    assert W.BRANCH_DTYPE.itemsize == 24 and W.MOUNT_DTYPE.itemsize == 20


def test_binding_constants_match_header():
    """Every TA_* value #defined in the header has the same value in the Python binding."""
    import re
    text = open(build.INCLUDE + "/treeattn.h").read()
    defs = dict(re.findall(r"#define\s+(TA_\w+)\s+\(?(-?(?:0x)?[0-9a-fA-F]+)u?\)?", text))
    assert len(defs) == len(re.findall(r"#define\s+TA_", text)) >= 11
    for name, val in defs.items():
        assert hasattr(_native, name), name
        assert getattr(_native, name) == int(val, 0), name
